// Receiver hot path: decode the frames of one window's stream and apply them
// in place to the receiver arena through the plan's canonical->receiver
// pieces, with per-chunk dedup, an overwrite-only retry mode, test-only fault
// injection and the commit check.
//
// Method: NeMo-DCR paper summary, "Recoverable in-place apply" (XOR masks
// flip the stored bits in place, overwrite records replace values, partial
// writes are retried, joint commit); popular write-up, sections on XOR versus
// overwrite, dedup by unique IDs, in-place apply without a backup copy and
// overwrite-only retry; "GPU-accelerated weight teleportation", "A strong
// baseline with the Blackwell-native DE" (one launch applies XOR to the whole
// model from a host-prepared plan) and "Working with low-precision RL" (the
// mask is remapped like the physical layout).
//
// Kernels (first phase: route_kernel, apply_kernel, lane_kernel, or
// apply_cta_kernel alone for plans of small windows; then, only
// when frames were deferred to them, defer_kernel and big_kernel; then the
// commit check):
//   route_kernel  one warp per 32 frames, a lane per frame: checks the index
//                 entry and frame header, claims the chunk (dedup) and lists
//                 the frame for the kernel that applies it.
//   apply_kernel  one warp per listed frame, 32 warps per SM.  XOR_RAW, OVERWRITE
//                 and OVERWRITE_DENSE frames are applied lane-parallel.  LZ4
//                 frames flagged ZSRC (every match copies zero bytes, as the
//                 library's encoder produces) have only literal bytes that can
//                 be non-zero, so nothing is materialised: lane 0 walks the
//                 tokens 32 sequences at a time, then the lanes XOR their
//                 sequences' non-zero literal bytes straight into the receiver
//                 arena and check every match against the sorted list of
//                 non-zero output bytes so far.  A frame that fails part-way is
//                 undone (XOR is self-inverse) before it is reported.
//   lane_kernel   one thread per ZSRC frame (streams of many frames): a
//                 serial walk that XORs the non-zero literal bytes and proves
//                 each match copies zeros from the zero stretches the
//                 library's encoder copies from; other frames to big_kernel.
//   big_kernel    one warp per ZSRC frame too large for apply_kernel's
//                 body cache or non-zero list (denser masks), and per ZSRC
//                 Snappy frame: the same walk (Snappy elements in place of
//                 LZ4 sequences) with the body read from global memory and
//                 the matches checked against a bitmap of the non-zero
//                 output bytes.  On plans of the Snappy codec, bodies up to
//                 8 KiB take the split walk instead: the lanes walk 32
//                 stretches of the body at once and join them (split_apply).
//   defer_kernel  one CTA per general LZ4 frame (any valid block, e.g. from
//                 the CPU oracle) or Snappy frame: full decode into a 64 KiB shared buffer
//                 with warp-parallel literal and match copies (a ZSRC frame
//                 whose match copies a non-zero byte is rejected), then the
//                 XOR sweep.
//   pending_kernel  counts framed chunks that are not DONE for the target
//                 version (the commit rule).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "dcr_internal.h"

namespace dcr {
namespace {

constexpr uint32_t kFull = 0xffffffffu;
constexpr int kAWarps = 16;                 // warps per CTA, one frame each; 2 CTAs per SM
constexpr int kAThreads = 32 * kAWarps;
constexpr int kBodyCache = 3072;            // bytes of LZ4 body cached per warp
constexpr int kAEvCap = 1024;               // non-zero output bytes listed per frame
constexpr int kDThreads = 256;
constexpr uint32_t kCasLimit = 1u << 16;

#include "decode.cuh"

struct ApplyArgs {
    const ChunkDesc* chunks;
    const Seg* dst;
    const uint64_t* win;
    uint32_t n_windows;
    int retry_only;
    const uint8_t* payload;
    uint64_t size;
    uint8_t* target;
    unsigned long long* state;
    ApplyScratch* sc;
    uint32_t* defer;          // deferred frames: general LZ4 from the front, large ZSRC from the back
    uint32_t* lane;           // ZSRC frames for lane_kernel (defer_len entries)
    uint32_t* warp;           // frames for apply_kernel (defer_len entries)
    uint32_t defer_len;
    uint64_t lane_min;        // frames in a stream from which lane_kernel takes its ZSRC frames
    int self_route;           // apply_kernel routes every frame itself (no route_kernel, no lane_kernel)
    int split_all;            // every ZSRC frame to big_kernel's split walk (DCR_APPLY_SPLIT)
    uint64_t plan_hash;
    uint64_t version;
    uint64_t abort_at;
    uint32_t split;
};

struct Hdr {
    uint64_t hash, base_v, target_v, n_frames, total, idx_off;
    uint32_t window, flags, chunk_begin, chunk_count;
};

constexpr uint32_t kWinA = 128;               // candidate sequence starts per walk window: apply_kernel
constexpr uint32_t kWinB = 160;               //                                          big_kernel
constexpr uint32_t kEndFinal = 0x80000000u;   // the sequence is the block's last
constexpr uint32_t kEndBad = 0x7FFFFFFFu;     // no valid sequence starts here
constexpr uint8_t kStop = 0xFF;               // jump: the chain stops (end, error, window left)

// one warp's shared memory: the frame body, the sorted positions of its
// non-zero output bytes so far, where a sequence starting at each byte of the
// current window would end, and the starts of one batch of sequences
struct __align__(16) AWarp {
    static constexpr uint32_t kWin = kWinA;
    uint8_t body[kBodyCache];
    uint16_t ev[kAEvCap];
    uint32_t nxt[kWin];
    uint32_t r_ip[32];
    uint8_t jmp[3][kWin];    // window-relative start 1, 2 and 4 sequences on, or kStop
    uint32_t base[8];
};

// big_kernel: one warp's shared memory.  Large ZSRC frames are read from
// global memory and their matches checked against a bitmap of the non-zero
// output bytes, which has no capacity limit.
struct __align__(16) BWarp {
    static constexpr uint32_t kWin = kWinB;   // denser masks: ~32 sequences per window
    static constexpr bool kSplit = false;
    static constexpr int kWarps = 8;
    uint32_t bits[kChunk / 32];
    uint32_t nxt[kWin];
    uint32_t r_ip[32];
    uint8_t jmp[3][kWin];
    uint32_t base[8];
};

// big_kernel on plans of the Snappy codec: bodies up to kSBody bytes are
// copied to shared memory and taken by the split walk (split_apply), which
// also keeps a bitmap of the element starts its lanes pass and the joins of
// the lanes' stretches; larger ones take the windowed walk.
constexpr uint32_t kSBody = 6144;
constexpr uint32_t kSChains = 4;   // walks per stretch, from its first four bytes
constexpr uint8_t kNoWalk = 0xFF;
struct __align__(16) SWarp {
    static constexpr uint32_t kWin = kWinB;
    static constexpr bool kSplit = true;
    static constexpr int kWarps = 5;
    union {
        uint32_t bits[kChunk / 32];            // the non-zero output bytes (both walks)
        uint8_t walker[kSBody];                // split walk, until the joins: per body byte, which walk of
                                               // its stretch passed an element start there (kNoWalk: none)
    };
    union {
        uint8_t body[kSBody + 16];             // split walk: the frame body (Walk::elem reads a byte past an element)
        struct {                               // windowed walk
            uint32_t nxt[kWin];
            uint32_t r_ip[32];
            uint8_t jmp[3][kWin];
            uint32_t base[8];
        };
    };
    uint32_t ex[32 * kSChains];                // split walk: where each walk leaves its stretch
    uint32_t T[33];                            // ... and the joins
};

struct __align__(16) ASmem {
    AWarp w[kAWarps];
    Hdr hdr;
    int ok;
};

__device__ __forceinline__ uint64_t ld64(const uint8_t* p)
{
    return *reinterpret_cast<const uint64_t*>(p);
}

__device__ __forceinline__ uint4 ld_nc16(const uint8_t* p)
{
    return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ bool is_zero(uint4 v) { return (v.x | v.y | v.z | v.w) == 0; }

// Stream header check, in the order: malformed -> plan/window mismatch ->
// retry-mode mismatch -> version mismatch.  Returns 0 or a dcr_status.
__device__ int check_header(const ApplyArgs& A, Hdr* h)
{
    const uint8_t* p = A.payload;
    uint32_t magic = *reinterpret_cast<const uint32_t*>(p);
    uint32_t fmt = *reinterpret_cast<const uint32_t*>(p + 4);
    h->hash = ld64(p + 8);
    h->base_v = ld64(p + 16);
    h->target_v = ld64(p + 24);
    h->window = *reinterpret_cast<const uint32_t*>(p + 32);
    h->flags = *reinterpret_cast<const uint32_t*>(p + 36);
    h->chunk_begin = *reinterpret_cast<const uint32_t*>(p + 40);
    h->chunk_count = *reinterpret_cast<const uint32_t*>(p + 44);
    h->n_frames = ld64(p + 48);
    h->total = ld64(p + 56);
    if (magic != kStreamMagic || fmt != kFormat || h->total > A.size || h->total < kStreamHdr ||
        h->total % 8 || h->n_frames > (h->total - kStreamHdr) / 8)
        return DCR_ERR_CORRUPT;
    h->idx_off = h->total - 8 * h->n_frames;
    if (h->hash != A.plan_hash || h->window >= A.n_windows ||
        h->chunk_begin != A.win[h->window] ||
        h->chunk_count != A.win[h->window + 1] - A.win[h->window])
        return DCR_ERR_INVALID;
    if (A.retry_only && !(h->flags & kStreamOverwriteOnly)) return DCR_ERR_INVALID;
    if (h->base_v != A.version) return DCR_ERR_VERSION;
    return 0;
}

__device__ __forceinline__ void report(ApplyScratch* sc, int code)
{
    atomicCAS(&sc->err, 0, code);
}

// receiver arena offset of canonical chunk byte x
__device__ __forceinline__ uint64_t dst_of(const Seg* s, uint32_t n, uint32_t x)
{
    if (n == 1) return s[0].addr + (x - s[0].off);
    int lo = 0, hi = int(n) - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (s[mid].off <= x) lo = mid;
        else hi = mid - 1;
    }
    return s[lo].addr + (x - s[lo].off);
}

// XOR one byte into the receiver: a fire-and-forget reduction on its 32-bit
// word (neighbouring bytes may belong to other frames' chunks)
__device__ __forceinline__ void xor_byte(uint8_t* target, uint64_t a, uint32_t b)
{
    const uintptr_t p = reinterpret_cast<uintptr_t>(target + a);
    asm volatile("red.global.xor.b32 [%0], %1;" ::"l"(p & ~uintptr_t(3)), "r"(b << (8 * (p & 3)))
                 : "memory");
}

// XOR one 16-byte mask vector at canonical chunk offset x (bytes >= lim skipped)
__device__ __forceinline__ void xor_vec(const ApplyArgs& A, const ChunkDesc& cd, const Seg* ds,
                                        uint32_t x, uint4 m, uint32_t lim)
{
    if ((cd.flags & kDstVec) && x + 16 <= lim) {
        uint4* d = reinterpret_cast<uint4*>(A.target + dst_of(ds, cd.dst_count, x));
        uint4 t = *d;
        *d = make_uint4(t.x ^ m.x, t.y ^ m.y, t.z ^ m.z, t.w ^ m.w);
        return;
    }
    const uint32_t w[4] = {m.x, m.y, m.z, m.w};
    for (int i = 0; i < 16; ++i) {
        uint32_t b = (w[i >> 2] >> (8 * (i & 3))) & 0xFFu;
        if (b && x + i < lim) xor_byte(A.target, dst_of(ds, cd.dst_count, x + i), b);
    }
}

__device__ __forceinline__ void put_vec(const ApplyArgs& A, const ChunkDesc& cd, const Seg* ds,
                                        uint32_t x, uint4 v, uint32_t lim, uint32_t raw)
{
    if ((cd.flags & kDstVec) && x + 16 <= lim) {
        *reinterpret_cast<uint4*>(A.target + dst_of(ds, cd.dst_count, x)) = v;
        return;
    }
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    for (int i = 0; i < 16; ++i)
        if (x + i < lim && x + i < raw)
            A.target[dst_of(ds, cd.dst_count, x + i)] = uint8_t(w[i >> 2] >> (8 * (i & 3)));
}

// claim a chunk for target version V: true if this frame may apply its mask
__device__ __forceinline__ bool claim(unsigned long long* st, uint64_t V, bool* timeout)
{
    unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(st);
    const unsigned long long want = (V << 2) | kClaimed;
    for (uint32_t i = 0; i < kCasLimit; ++i) {
        if ((cur >> 2) == V && (cur & 3) != kNotStarted) return false;
        unsigned long long seen = atomicCAS(st, cur, want);
        if (seen == cur) return true;
        cur = seen;
    }
    *timeout = true;
    return false;
}

// XOR is its own inverse: re-applying the first `runs` literal runs of a frame
// that failed part-way restores every byte the failed pass touched, so a
// corrupt frame leaves its chunk exactly as it was (the overwrite-only retry
// rewrites changed units only and could not repair bytes outside them).  The
// runs replayed passed every bounds check the first time.
__device__ void zsrc_undo(const ApplyArgs& A, const ChunkDesc& cd, const Seg* ds,
                          const uint8_t* src, uint32_t lim, uint32_t runs, int lane)
{
    uint32_t ip = 0, op = 0;
    for (uint32_t r = 0; r < runs; ++r) {
        const uint32_t tok = src[ip++];
        uint32_t ll = tok >> 4;
        if (ll == 15) {
            uint32_t b;
            do {
                b = src[ip++];
                ll += b;
            } while (b == 255);
        }
        for (uint32_t i = lane; i < ll; i += 32) {
            uint32_t b = src[ip + i];
            uint32_t x = op + i;
            if (b && x < lim) xor_byte(A.target, dst_of(ds, cd.dst_count, x), b);
        }
        __syncwarp();
        ip += ll;
        op += ll;
        if (r + 1 == runs) break;
        ip += 2;
        uint32_t ml = tok & 15u;
        if (ml == 15) {
            uint32_t b;
            do {
                b = src[ip++];
                ml += b;
            } while (b == 255);
        }
        op += ml + 4;
    }
}

__device__ __forceinline__ uint32_t warp_incl_sum(uint32_t v, int lane)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_up_sync(kFull, v, d);
        if (lane >= d) v += o;
    }
    return v;
}

// ---- ZSRC frames: chained walk, parallel apply ---------------------------
// End of the sequence starting at body byte p (where the next one starts),
// | kEndFinal for a literals-only last sequence, or kEndBad.
__device__ __forceinline__ uint32_t seq_end(const uint8_t* src, uint32_t n, uint32_t p)
{
    if (p >= n) return kEndBad;
    const uint32_t tok = src[p];
    uint32_t q = p + 1, ll = tok >> 4;
    if (ll == 15) {
        uint32_t b;
        do {
            if (q >= n) return kEndBad;
            b = src[q++];
            ll += b;
        } while (b == 255);
    }
    if (ll > n - q) return kEndBad;
    q += ll;
    if (q == n) return q | kEndFinal;
    if (n - q < 2) return kEndBad;
    q += 2;
    if ((tok & 15u) == 15u) {
        uint32_t b;
        do {
            if (q >= n) return kEndBad;
            b = src[q++];
        } while (b == 255);
    }
    return q;
}

__device__ __noinline__ uint32_t seq_end_rare(const uint8_t* src, uint32_t n, uint32_t p)
{
    return seq_end(src, n, p);
}

// seq_end for a body in global memory: the common shape (literal length
// below 15, at most one match-length byte, below 255) without branches, both
// bytes it may need read at once, clamped into the body (n >= 1).
__device__ __forceinline__ uint32_t seq_end_ldg(const uint8_t* src, uint32_t n, uint32_t p)
{
    const uint32_t tok = src[p < n ? p : n - 1];
    const uint32_t ll = tok >> 4;
    const uint32_t q = p + 1 + ll;   // end of the literals
    const uint32_t x = src[q + 2 < n ? q + 2 : n - 1];
    const bool mlx = (tok & 15u) == 15u;
    if (p >= n) return kEndBad;
    if (ll == 15 || (mlx && x == 255)) return seq_end_rare(src, n, p);
    if (q > n) return kEndBad;
    if (q == n) return q | kEndFinal;
    if (n - q < 2 || (mlx && n - q < 3)) return kEndBad;
    return q + (mlx ? 3u : 2u);
}

// How zsrc_apply reads a block: where its first element starts, where the
// element starting at body byte p ends (| kEndFinal when the block ends
// there, kEndBad when no valid element starts at p), an element's literal
// run and match (off, ml; ml == 0: none), and how to replay the literal runs
// of a frame's first elements (undo).
//
// LZ4 ("A strong baseline with the Blackwell-native DE": the LZ4 block
// format): a sequence is a token, its literals, a 2-byte offset and the
// match-length bytes; the last sequence is literals only.
struct Lz4Walk {
    static constexpr uint32_t kWin = 256;   // no limit below the warp's window
    __device__ static uint32_t first(const uint8_t*, uint32_t, uint32_t) { return 0; }
    template <bool kGlobal>
    __device__ static uint32_t end(const uint8_t* src, uint32_t n, uint32_t p)
    {
        return kGlobal ? seq_end_ldg(src, n, p) : seq_end(src, n, p);
    }
    __device__ static void decode(const uint8_t* src, uint32_t q, bool last, uint32_t& ipl, uint32_t& ll,
                                  uint32_t& off, uint32_t& ml)
    {
        const uint32_t tok = src[q++];
        ll = tok >> 4;
        if (ll == 15) {
            uint32_t b;
            do {
                b = src[q++];
                ll += b;
            } while (b == 255);
        }
        ipl = q;
        q += ll;
        off = ml = 0;
        if (!last) {
            off = uint32_t(src[q]) | (uint32_t(src[q + 1]) << 8);
            q += 2;
            ml = tok & 15u;
            if (ml == 15) {
                uint32_t b;
                do {
                    b = src[q++];
                    ml += b;
                } while (b == 255);
            }
            ml += 4;
        }
    }
    __device__ static void undo(const ApplyArgs& A, const ChunkDesc& cd, const Seg* ds, const uint8_t* src, uint32_t,
                                uint32_t, uint32_t lim, uint32_t runs, int lane)
    {
        zsrc_undo(A, cd, ds, src, lim, runs, lane);
    }
    // one sequence at p whose bounds end() has checked: its fields and where
    // the next starts (| kEndFinal after the block's last)
    __device__ static uint32_t elem(const uint8_t* src, uint32_t n, uint32_t p, uint32_t& ipl, uint32_t& ll,
                                    uint32_t& off, uint32_t& ml)
    {
        const uint32_t tok = src[p];
        uint32_t q = p + 1;
        ll = tok >> 4;
        if (ll == 15) {
            uint32_t b;
            do {
                b = src[q++];
                ll += b;
            } while (b == 255);
        }
        ipl = q;
        q += ll;
        off = ml = 0;
        if (q == n) return q | kEndFinal;
        off = uint32_t(src[q]) | (uint32_t(src[q + 1]) << 8);
        q += 2;
        ml = tok & 15u;
        if (ml == 15) {
            uint32_t b;
            do {
                b = src[q++];
                ml += b;
            } while (b == 255);
        }
        ml += 4;
        return q;
    }
};

// Snappy (the same section, footnote 4): a varint of the output length, then
// literal elements (tag (length - 1) << 2, or 60..63 and 1..4 length bytes)
// and copies (tag 1: length 4..11, 11-bit offset; tag 2 / 3: length 1..64,
// 2- / 4-byte offset).  An element is a literal run or a copy.
struct SnappyWalk {
    // elements average under 3 bytes: 96 bytes hold the 32 a batch takes
    static constexpr uint32_t kWin = 96;
    __device__ static uint32_t first(const uint8_t* src, uint32_t n, uint32_t raw)
    {
        uint64_t v = 0;
        uint32_t ip = 0;
        for (uint32_t shift = 0; shift <= 28 && ip < n; shift += 7) {
            const uint64_t b = src[ip++];
            v |= (b & 127u) << shift;
            if (!(b & 128u)) return v == raw ? ip : kEndBad;
        }
        return kEndBad;
    }
    // end() of a literal with 1..4 length bytes
    __device__ static __noinline__ uint32_t end_long(const uint8_t* src, uint32_t n, uint32_t p)
    {
        const uint32_t nb = (src[p] >> 2) - 59;
        if (uint64_t(p) + 1 + nb > n) return kEndBad;
        uint64_t len = 0;
        for (uint32_t i = 0; i < nb; ++i) len |= uint64_t(src[p + 1 + i]) << (8 * i);
        const uint64_t e = uint64_t(p) + 1 + nb + len + 1;
        if (e > n) return kEndBad;
        return e == n ? uint32_t(e) | kEndFinal : uint32_t(e);
    }
    template <bool>
    __device__ static uint32_t end(const uint8_t* src, uint32_t n, uint32_t p)
    {
        if (p >= n) return kEndBad;
        const uint32_t tag = src[p], t = tag & 3u;
        if (t != 0 || tag < 240u) {   // a copy (2, 3 or 5 bytes) or a literal of up to 60 bytes
            const uint32_t e = p + (t ? (0x5320u >> (4 * t)) & 15u : 2u + (tag >> 2));
            if (e > n) return kEndBad;
            return e == n ? e | kEndFinal : e;
        }
        return end_long(src, n, p);
    }
    __device__ static void decode(const uint8_t* src, uint32_t q, bool, uint32_t& ipl, uint32_t& ll, uint32_t& off,
                                  uint32_t& ml)
    {
        const uint32_t tag = src[q], t = tag & 3u;
        if (t == 0) {
            uint32_t len = (tag >> 2) + 1, nb = 0;
            if ((tag >> 2) >= 60) {
                nb = (tag >> 2) - 59;
                len = 0;
                for (uint32_t i = 0; i < nb; ++i) len |= uint32_t(src[q + 1 + i]) << (8 * i);
                len += 1;
            }
            ll = len;
            ipl = q + 1 + nb;
            off = ml = 0;
        } else {
            ll = 0;
            ipl = q;
            if (t == 1) {
                ml = ((tag >> 2) & 7u) + 4;
                off = ((tag >> 5) << 8) | src[q + 1];
            } else {
                ml = (tag >> 2) + 1;
                off = 0;
                for (uint32_t i = 0; i < (t == 2 ? 2u : 4u); ++i) off |= uint32_t(src[q + 1 + i]) << (8 * i);
            }
        }
    }
    // one element at p whose bounds end() has checked: its fields and where
    // the next starts (| kEndFinal after the block's last)
    __device__ static uint32_t elem(const uint8_t* src, uint32_t n, uint32_t p, uint32_t& ipl, uint32_t& ll,
                                    uint32_t& off, uint32_t& ml)
    {
        const uint32_t tag = src[p], t = tag & 3u;
        uint32_t q;
        if (t == 0 && tag >= 240u) {   // a literal with 1..4 length bytes
            const uint32_t nb = (tag >> 2) - 59;
            uint32_t len = 0;
            for (uint32_t i = 0; i < nb; ++i) len |= uint32_t(src[p + 1 + i]) << (8 * i);
            ipl = p + 1 + nb;
            ll = len + 1;
            off = ml = 0;
            q = ipl + ll;
        } else {
            // the other shapes without branches; the element holds at least
            // two bytes, and for copies of one offset byte the second one
            // read belongs to the next element or to the buffer's padding
            // (unused)
            const uint32_t b1 = src[p + 1], b2 = src[p + 2];
            const bool lit = t == 0;
            ipl = p + (lit ? 1u : 0u);
            ll = lit ? (tag >> 2) + 1 : 0u;
            ml = lit ? 0u : t == 1 ? ((tag >> 2) & 7u) + 4 : (tag >> 2) + 1;
            off = lit ? 0u : t == 1 ? ((tag >> 5) << 8) | b1 : b1 | (b2 << 8);
            q = lit ? p + 1 + ll : p + ((0x5320u >> (4 * t)) & 15u);
            if (t == 3) off |= (uint32_t(src[p + 3]) << 16) | (uint32_t(src[p + 4]) << 24);
        }
        return q == n ? q | kEndFinal : q;
    }
    __device__ static void undo(const ApplyArgs& A, const ChunkDesc& cd, const Seg* ds, const uint8_t* src, uint32_t n,
                                uint32_t raw, uint32_t lim, uint32_t runs, int lane)
    {
        uint32_t q = first(src, n, raw), o = 0;
        for (uint32_t r = 0; r < runs; ++r) {
            uint32_t ipl, ll, off, ml;
            decode(src, q, false, ipl, ll, off, ml);
            for (uint32_t i = lane; i < ll; i += 32) {
                const uint32_t b = src[ipl + i], x = o + i;
                if (b && x < lim) xor_byte(A.target, dst_of(ds, cd.dst_count, x), b);
            }
            __syncwarp();
            o += ll + ml;
            q = end<true>(src, n, q) & ~kEndFinal;
        }
    }
};

// The warp takes the block a window of kWin body bytes at a time (WS::kWin:
// 128 for apply_kernel, 160 for the denser frames of big_kernel): every lane
// works out where a sequence starting at each of its window bytes would end
// (and, in two more passes, where the sequence two and four on starts), lane
// 0 follows the chain from the current sequence four sequences per shared
// load, and up to 32 sequences found that way are decoded one per lane, their
// output positions given by a warp prefix sum.  Then each
// lane XORs the non-zero literal bytes of its sequence into the receiver,
// lists their positions (the warp's list of non-zero output bytes stays
// sorted, since literal runs come in output order), and checks that its
// match copies zero bytes only: no listed position falls in the match's
// source range.  Returns 1 if the frame was applied, 0 if it is malformed or
// breaks its ZSRC promise, 2 if it holds more non-zero bytes than the list
// (the caller defers it); in the last two cases the partial apply has been
// undone.
//
// kBitmap (big_kernel): the non-zero output bytes are kept as a bitmap over
// the chunk instead of a sorted list, so there is no capacity limit, and src
// may be the frame body in global memory.
template <bool kBitmap, class WS, class Walk = Lz4Walk>
__device__ int zsrc_apply(const ApplyArgs& A, const ChunkDesc& cd, const Seg* ds, const uint8_t* src,
                          uint32_t n, uint32_t raw, uint32_t lim, WS& W, int lane)
{
    if (n == 0) return 0;   // a block holds at least one element
    const uint32_t ip0 = Walk::first(src, n, raw);
    if (ip0 == kEndBad) return 0;
    constexpr uint32_t kWin = Walk::kWin < WS::kWin ? Walk::kWin : WS::kWin;
    static_assert(kWin % 32 == 0 && kWin < kStop, "window: whole lane groups, offsets below kStop");
    const bool one = cd.dst_count == 1;
    const uint64_t base = one ? ds[0].addr - ds[0].off : 0ull;   // single receiver piece
    if constexpr (kBitmap) {
        for (uint32_t w = lane; w < (raw + 31) / 32; w += 32) W.bits[w] = 0;
        __syncwarp();
    }
    uint32_t ip = ip0, op = 0;    // next sequence in the body; its output position
    uint32_t nev = 0, runs = 0;   // listed positions, literal runs applied
    uint32_t cs = 0, ce = 0;      // output bytes [cs, ce) known to be zero
    int status = 1;
    for (;;) {
        uint32_t e[kWin / 32];
#pragma unroll
        for (uint32_t j = 0; j < kWin / 32; ++j)
            e[j] = Walk::template end<kBitmap>(src, n, ip + 32 * j + lane);
#pragma unroll
        for (uint32_t j = 0; j < kWin / 32; ++j) {
            const uint32_t x = e[j];
            W.nxt[32 * j + lane] = x;
            W.jmp[0][32 * j + lane] =
                (x == kEndBad || (x & kEndFinal) || x >= n || x - ip >= kWin) ? kStop : uint8_t(x - ip);
        }
        __syncwarp();
        // two and four sequences on, for every window byte
#pragma unroll
        for (int t = 1; t < 3; ++t) {
            uint8_t y[kWin / 32];
#pragma unroll
            for (uint32_t j = 0; j < kWin / 32; ++j) {
                const uint8_t a = W.jmp[t - 1][32 * j + lane];
                y[j] = a == kStop ? kStop : W.jmp[t - 1][a];
            }
#pragma unroll
            for (uint32_t j = 0; j < kWin / 32; ++j) W.jmp[t][32 * j + lane] = y[j];
            __syncwarp();
        }
        // lane 0 follows the chain four sequences at a time, then one at a
        // time for its last few; the other lanes fill in the skipped starts
        uint32_t nb = 0, cnt = 0, fin = 0, bad = 0, cur = ip;
        if (lane == 0) {
            uint32_t p = 0;
            while (nb < 8 && W.jmp[2][p] != kStop) {
                W.base[nb++] = p;
                p = W.jmp[2][p];
            }
            cnt = 4 * nb;
            if (nb == 8) {
                cur = ip + p;
            } else {
                for (int t = 0; t < 4; ++t) {
                    const uint32_t x = W.nxt[p];
                    if (x == kEndBad) { bad = 1; break; }
                    W.r_ip[cnt++] = ip + p;
                    if (x & kEndFinal) { fin = 1; cur = x & ~kEndFinal; break; }
                    if (x >= n) { bad = 1; break; }   // a block ends with a literals-only sequence
                    if (x - ip >= kWin) { cur = x; break; }
                    p = x - ip;
                }
            }
        }
        nb = __shfl_sync(kFull, nb, 0);
        cnt = __shfl_sync(kFull, cnt, 0);
        fin = __shfl_sync(kFull, fin, 0);
        bad = __shfl_sync(kFull, bad, 0);
        cur = __shfl_sync(kFull, cur, 0);
        __syncwarp();
        if (lane < int(4 * nb)) {
            const uint32_t b = W.base[lane >> 2];
            const uint32_t k = lane & 3;
            const uint32_t q = k == 0 ? b : k == 1 ? W.jmp[0][b] : k == 2 ? W.jmp[1][b] : W.jmp[0][W.jmp[1][b]];
            W.r_ip[lane] = ip + q;
        }
        if (bad) {
            status = 0;
            break;
        }
        __syncwarp();
        // one sequence per lane (its bytes were bounds-checked by seq_end)
        const bool mine = lane < int(cnt);
        const bool lastseq = fin && lane == int(cnt) - 1;
        uint32_t ipl = 0, ll = 0, off = 0, ml = 0;
        if (mine) Walk::decode(src, W.r_ip[lane], lastseq, ipl, ll, off, ml);
        const uint32_t len = ll + ml;
        const uint32_t lincl = warp_incl_sum(len, lane);
        const uint32_t opl = op + lincl - len;   // output position of the literals
        const uint32_t mop = opl + ll;           // ... and of the match
        bool wrong = false;
        if (mine) {
            wrong = opl > raw || ll > raw - opl;
            if (ml) wrong = wrong || off == 0 || off > mop || ml > raw - mop;
            if (lastseq) wrong = wrong || mop + ml != raw;   // the block ends exactly at the chunk's end
        }
        if (__any_sync(kFull, wrong)) {
            status = 0;
            break;
        }
        op += __shfl_sync(kFull, lincl, 31);
        ip = cur;
        // literals: XOR into the receiver and record the non-zero ones
        if constexpr (kBitmap) {
            // the first four literal bytes are read at once (clamped into
            // the body), the rest one by one
            for (uint32_t q = 0; q < ll; ++q) {
                const uint32_t b = src[ipl + q];
                if (b) {
                    const uint32_t x = opl + q;
                    atomicOr(&W.bits[x >> 5], 1u << (x & 31));
                    if (x < lim) xor_byte(A.target, one ? base + x : dst_of(ds, cd.dst_count, x), b);
                }
            }
        } else {
            uint32_t c = 0;
            for (uint32_t q = 0; q < ll; ++q) c += src[ipl + q] != 0;
            const uint32_t incl = warp_incl_sum(c, lane);
            const uint32_t tot = __shfl_sync(kFull, incl, 31);
            if (nev + tot > uint32_t(kAEvCap)) {
                status = 2;
                break;
            }
            uint32_t at = nev + incl - c;
            for (uint32_t q = 0; q < ll; ++q) {
                const uint32_t b = src[ipl + q];
                if (b) {
                    const uint32_t x = opl + q;
                    W.ev[at++] = uint16_t(x);
                    if (x < lim) xor_byte(A.target, one ? base + x : dst_of(ds, cd.dst_count, x), b);
                }
            }
            nev += tot;
        }
        runs += cnt;
        __syncwarp();
        // the match copies [mop - off, mop - off + min(ml, off)), repeated
        bool viol = false;
        if constexpr (kBitmap) {
            if (mine && ml) {
                const uint32_t s0 = mop - off, e0 = s0 + (ml < off ? ml : off);
                for (uint32_t w = s0 >> 5; w <= (e0 - 1) >> 5 && !viol; ++w) {
                    const uint32_t a = (w << 5) > s0 ? 0u : s0 - (w << 5);
                    const uint32_t b = ((w + 1) << 5) < e0 ? 32u : e0 - (w << 5);
                    const uint32_t m = (b == 32 ? 0xFFFFFFFFu : ((1u << b) - 1)) & ~((1u << a) - 1);
                    viol = (W.bits[w] & m) != 0;
                }
            }
        } else {
            // a source inside the sequence's own literals (offset 1 after a
            // kept zero) is checked there, one inside [cs, ce) needs no check,
            // the rest are looked up in the list; the longest zero stretch
            // found that way is kept
            bool look = false;
            uint32_t s0 = 0, e0 = 0, zs = 0, ze = 0;
            if (mine && ml) {
                s0 = mop - off;
                e0 = s0 + (ml < off ? ml : off);
                if (off <= ll && e0 - s0 <= 4u) {
                    for (uint32_t q = ll - off; q < ll - off + (e0 - s0); ++q) viol |= src[ipl + q] != 0;
                } else {
                    look = s0 < cs || e0 > ce;
                }
            }
            if (__any_sync(kFull, look)) {
                if (look) {
                    uint32_t lo = 0, hi = nev;   // first listed position >= s0
                    while (lo < hi) {
                        const uint32_t mid = (lo + hi) >> 1;
                        if (W.ev[mid] < s0) lo = mid + 1;
                        else hi = mid;
                    }
                    viol = lo < nev && W.ev[lo] < e0;
                    // the zero stretch between the listed neighbours (every
                    // non-zero output byte before op is listed)
                    zs = lo ? uint32_t(W.ev[lo - 1]) + 1u : 0u;
                    ze = lo < nev ? uint32_t(W.ev[lo]) : op;
                }
                const uint32_t zl = look && !viol ? ze - zs : 0u;
                const uint32_t best = __reduce_max_sync(kFull, zl);
                if (best > ce - cs) {
                    const int from = __ffs(__ballot_sync(kFull, zl == best)) - 1;
                    cs = __shfl_sync(kFull, zs, from);
                    ce = __shfl_sync(kFull, ze, from);
                }
            }
        }
        if (__reduce_or_sync(kFull, uint32_t(viol))) {
            status = 0;
            break;
        }
        if (fin) break;
        __syncwarp();   // the window and the batch are rewritten
    }
    if (status != 1 && runs) Walk::undo(A, cd, ds, src, n, raw, lim, runs, lane);
    return status;
}

// The split walk.  A chain of elements (LZ4 sequences or Snappy elements) is
// a function of where it starts: two walks that meet at one start go on
// together.  So the body after the block's preamble is cut into 32 stretches
// of equal length, one per lane, and every lane walks its stretch at once
// from each of its first four bytes as though an element started there
// (a walk that meets one of the lane's earlier walks stops, as it would go
// on the same way), marking the starts it passes and which walk passed them;
// lane 0's first walk starts at the block's first element and is the true
// one.  Four walks, since in the runs of equal short elements the library's
// encoder writes a walk that starts inside an element can stay out of step
// with the true chain.  Lane 0 then joins the stretches in order: the true
// chain enters stretch i where the walk of stretch i - 1 leaves it, and from
// the first start there that lane i marked it is that walk of lane i's, so
// only the elements before that join are walked again.  Every element of the
// chain has passed the bounds checks of Walk::end once this is done, and a
// chain that does not end with the block's last element exactly at the end
// of the body is rejected before anything is written.  Each lane then takes
// the true elements that start in its stretch: it sums their output lengths
// (a warp prefix sum gives its first output position; the sum must be the
// chunk's length), XORs their non-zero literal bytes into the receiver while
// marking them in a bitmap of the chunk, and, once every lane has marked its
// literals, checks that each match or copy reads only unmarked bytes below
// its own position: all other output bytes are copies of zeros.  A frame that
// breaks that promise is undone by XORing the same literal bytes again.
// src is the body in shared memory (n <= kSBody); 1 if the frame was applied,
// 0 if it is malformed or lying (nothing of it left applied).
template <class Walk, class WS>
__device__ int split_apply(const ApplyArgs& A, const ChunkDesc& cd, const Seg* ds, const uint8_t* src, uint32_t n,
                           uint32_t raw, uint32_t lim, WS& W, int lane)
{
    if (n == 0) return 0;
    const uint32_t ip0 = Walk::first(src, n, raw);
    if (ip0 >= n) return 0;   // kEndBad too; a block holds at least one element
    const uint32_t span = n - ip0, S = (span + 31) / 32;
    auto edge = [&](uint32_t i) { return ip0 + (i * S < span ? i * S : span); };   // stretch i is [edge(i), edge(i + 1))
    const uint32_t s0 = edge(lane), s1 = edge(lane + 1);
    auto bad_end = [&](uint32_t x) { return x == kEndBad || (!(x & kEndFinal) && x >= n); };
    for (uint32_t v = lane; v < (n + 15) / 16; v += 32)
        reinterpret_cast<uint4*>(W.walker)[v] = make_uint4(~0u, ~0u, ~0u, ~0u);
    __syncwarp();
    // 1. the lane's walks of its stretch; a walk's exit is the first start at
    //    or past the stretch's end, the block's end | kEndFinal, or kEndBad
    //    (one element per round, the lane's walks one after another)
    {
        uint32_t c = 0, p = s0;
        while (c < kSChains) {
            uint32_t ex = 0;
            bool done = true;
            const uint32_t by = p < s1 ? W.walker[p] : kNoWalk;
            if (p >= s1) {
                ex = s1;   // a stretch shorter than its walks
            } else if (by != kNoWalk) {   // an earlier walk of this lane passed p: the same from here
                ex = W.ex[kSChains * lane + by];
            } else {
                W.walker[p] = uint8_t(c);
                const uint32_t x = Walk::template end<false>(src, n, p);
                if (bad_end(x)) ex = kEndBad;
                else if ((x & kEndFinal) || x >= s1) ex = x;
                else {
                    p = x;
                    done = false;
                }
            }
            if (done) {
                W.ex[kSChains * lane + c] = ex;
                ++c;
                p = s0 + c;
            }
        }
    }
    __syncwarp();
    // 2. the joins: T[i] is the first true start at or past edge(i) (or the
    //    chain's end), T[32] the chain's end
    if (lane == 0) {
        uint32_t t = W.ex[0];
        W.T[0] = ip0;
        for (uint32_t i = 1; i < 32; ++i) {
            W.T[i] = t;
            const uint32_t b = edge(i + 1);
            if (t == kEndBad || (t & kEndFinal) || t >= b) continue;
            for (uint32_t q = t;;) {
                const uint32_t by = W.walker[q];
                if (by != kNoWalk) {   // joined one of lane i's walks
                    t = W.ex[kSChains * i + by];
                    break;
                }
                const uint32_t x = Walk::template end<false>(src, n, q);
                if (bad_end(x)) {
                    t = kEndBad;
                    break;
                }
                if ((x & kEndFinal) || x >= b) {
                    t = x;
                    break;
                }
                q = x;
            }
        }
        W.T[32] = t;
    }
    __syncwarp();
    if (W.T[32] != (n | kEndFinal)) return 0;
    // this lane's true elements: those that start in [T[lane], s1), each
    // bounds-checked by Walk::end in step 1 or 2
    const uint32_t t0 = W.T[lane];
    auto walk = [&](auto&& fn) {
        if (t0 & kEndFinal) return;   // (kEndBad cannot occur past a good chain)
        for (uint32_t p = t0; p < s1;) {
            uint32_t ipl, ll, off, ml;
            const uint32_t x = Walk::elem(src, n, p, ipl, ll, off, ml);
            fn(ipl, ll, off, ml);
            if (x & kEndFinal) break;
            p = x;
        }
    };
    // 3. output positions
    uint32_t len = 0;
    walk([&](uint32_t, uint32_t ll, uint32_t, uint32_t ml) { len += ll + ml; });
    const uint32_t incl = warp_incl_sum(len, lane);
    if (__shfl_sync(kFull, incl, 31) != raw) return 0;
    const uint32_t op0 = incl - len;
    // 4. literals: XOR the non-zero bytes into the receiver (mark: and into
    //    the bitmap); every output position is below raw
    for (uint32_t v = lane; v < (raw + 127) / 128; v += 32) reinterpret_cast<uint4*>(W.bits)[v] = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();
    const bool one = cd.dst_count == 1;
    const uint64_t base = one ? ds[0].addr - ds[0].off : 0ull;
    auto literals = [&](bool mark) {
        uint32_t op = op0;
        walk([&](uint32_t ipl, uint32_t ll, uint32_t, uint32_t ml) {
            for (uint32_t q = 0; q < ll; ++q) {
                const uint32_t b = src[ipl + q];
                if (b) {
                    const uint32_t x = op + q;
                    if (mark) atomicOr(&W.bits[x >> 5], 1u << (x & 31));
                    if (x < lim) xor_byte(A.target, one ? base + x : dst_of(ds, cd.dst_count, x), b);
                }
            }
            op += ll + ml;
        });
    };
    literals(true);
    __syncwarp();
    // 5. every match or copy reads [mop - off, mop - off + min(ml, off)),
    //    repeated: no marked byte may fall there
    bool viol = false;
    {
        uint32_t op = op0;
        const uint32_t nw = (raw + 31) / 32;
        walk([&](uint32_t, uint32_t ll, uint32_t off, uint32_t ml) {
            const uint32_t mop = op + ll;
            op = mop + ml;
            // literal runs (ml = 0) check nothing: L = 0
            const bool good = off != 0 && off <= mop;
            viol |= ml != 0 && !good;
            const uint32_t a0 = good ? mop - off : 0u, L = ml == 0 || !good ? 0u : ml < off ? ml : off;
            if (L <= 64) {   // the 64 bits from a0 on, from three words (past the chunk: none)
                const uint32_t w = a0 >> 5, sh = a0 & 31;
                const uint64_t lo = uint64_t(W.bits[w]) | (w + 1 < nw ? uint64_t(W.bits[w + 1]) << 32 : 0ull);
                uint64_t v = lo >> sh;
                if (sh && w + 2 < nw) v |= uint64_t(W.bits[w + 2]) << (64 - sh);
                viol |= (v & (L == 64 ? ~0ull : (1ull << L) - 1)) != 0;
            } else {
                const uint32_t e0 = a0 + L;
                for (uint32_t w = a0 >> 5; w <= (e0 - 1) >> 5 && !viol; ++w) {
                    const uint32_t a = (w << 5) > a0 ? 0u : a0 - (w << 5);
                    const uint32_t b = ((w + 1) << 5) < e0 ? 32u : e0 - (w << 5);
                    const uint32_t m = (b == 32 ? 0xFFFFFFFFu : ((1u << b) - 1)) & ~((1u << a) - 1);
                    viol = (W.bits[w] & m) != 0;
                }
            }
        });
    }
    if (__any_sync(kFull, viol)) {
        literals(false);   // XOR is its own inverse
        return 0;
    }
    return 1;
}

// ================================================================ kernels ==
// Where apply_kernel sends a frame.
enum FrameRoute : int { kRNone = 0, kRSkip, kRWarp, kRDefer, kRLane, kRBig };

// One lane's part of apply_kernel: check frame f's index entry and header
// (errors reported), skip it past an injected fault, claim its chunk (XOR
// kinds; kRSkip: already claimed or done for this version), and route it:
// general LZ4 and Snappy frames to the full decode; ZSRC frames to
// lane_kernel when the stream has frames enough to keep its threads busy,
// else Snappy ones and LZ4 ones larger than the body cache to big_kernel;
// the rest to the warp.
__device__ __forceinline__ int frame_route(const ApplyArgs& A, const Hdr& H, uint32_t f)
{
    const uint64_t fo = ld64(A.payload + H.idx_off + 8ull * f);
    if (fo < kStreamHdr || fo % 16 || fo + kFrameHdr > H.idx_off) {
        report(A.sc, DCR_ERR_CORRUPT);
        return kRNone;
    }
    const uint4 h0 = ld_nc16(A.payload + fo), h1 = ld_nc16(A.payload + fo + 16);
    const uint32_t kind = h0.y & 0xFFu, fbits = (h0.y >> 8) & 0xFFu, fflags = h0.y >> 16;
    const uint32_t c = h0.z, raw = h0.w, bl = h1.x;
    if (h0.x != kFrameMagic || kind < kXorLz4 || kind > kXorSnappy || c < H.chunk_begin ||
        c >= H.chunk_begin + H.chunk_count || bl > H.idx_off - fo - kFrameHdr) {
        report(A.sc, DCR_ERR_CORRUPT);
        return kRNone;
    }
    const ChunkDesc cd = A.chunks[c];
    if (raw != cd.raw_len || fbits != cd.bits) {
        report(A.sc, DCR_ERR_CORRUPT);
        return kRNone;
    }
    const bool is_xor = kind == kXorLz4 || kind == kXorRaw || kind == kXorSnappy;
    if (A.retry_only && is_xor) {
        report(A.sc, DCR_ERR_INVALID);
        return kRNone;
    }
    if (uint64_t(f) > A.abort_at) return kRNone;   // injected fault: never reached
    if (!is_xor) return kRWarp;
    bool to = false;
    if (!claim(&A.state[c], H.target_v, &to)) {
        if (to) report(A.sc, DCR_ERR_TIMEOUT);
        return to ? kRNone : kRSkip;
    }
    const bool zs = (fflags & kFrameZsrc) != 0;
    if (kind != kXorRaw && !zs) return kRDefer;
    if (kind != kXorRaw && A.split_all) return kRBig;
    if (kind != kXorRaw && H.n_frames >= A.lane_min) return kRLane;
    if (kind == kXorSnappy || (kind == kXorLz4 && bl > uint32_t(kBodyCache))) return kRBig;
    return kRWarp;
}

// The warp's frames routed to list r, appended with one atomic per warp.
__device__ __forceinline__ void push_listed(const ApplyArgs& A, int route, int r, uint32_t f, int lane,
                                            uint32_t lt)
{
    const uint32_t m = __ballot_sync(kFull, route == r);
    if (!m) return;
    uint32_t* cnt = r == kRDefer ? &A.sc->n_defer : r == kRLane ? &A.sc->n_lane
                  : r == kRBig ? &A.sc->n_big : &A.sc->n_warp;
    uint32_t base = 0;
    if (lane == 0) base = atomicAdd(cnt, uint32_t(__popc(m)));
    base = __shfl_sync(kFull, base, 0);
    if (route != r) return;
    const uint32_t k = base + __popc(m & lt);
    if (r == kRDefer) A.defer[k] = f;
    else if (r == kRLane) A.lane[k] = f;
    else if (r == kRBig) A.defer[A.defer_len - 1 - k] = f;
    // a well-formed stream holds one frame per chunk and claimed frames
    // never outnumber the chunks; only repeated overwrite frames (applied
    // unclaimed) can: more than the list holds is rejected
    else if (k < A.defer_len) A.warp[k] = f;
    else report(A.sc, DCR_ERR_CORRUPT);
}

// The first apply kernel of the warp route: one warp per 32 frames, each
// lane checks, claims and routes one frame (frame_route) into the lists of
// the kernels after it: apply_kernel, lane_kernel, defer_kernel, big_kernel.
constexpr int kRtThreads = 256;

__global__ void __launch_bounds__(kRtThreads) route_kernel(ApplyArgs A)
{
    __shared__ Hdr hdr;
    __shared__ int ok;
    if (threadIdx.x == 0) {
        const int rc = check_header(A, &hdr);
        ok = rc == 0;
        if (rc) report(A.sc, rc);
        else if (blockIdx.x == 0) {
            A.sc->hdr_ok = 1;
            A.sc->target_version = hdr.target_v;
            A.sc->window = hdr.window;
            A.sc->n_frames = hdr.n_frames;
        }
    }
    __syncthreads();
    if (!ok) return;
    const Hdr H = hdr;
    const int lane = threadIdx.x & 31;
    const uint32_t lt = (1u << lane) - 1u;
    const uint64_t nw = uint64_t(gridDim.x) * (kRtThreads / 32);
    for (uint64_t f0 = 32 * (uint64_t(blockIdx.x) * (kRtThreads / 32) + (threadIdx.x >> 5)); f0 < H.n_frames;
         f0 += 32 * nw) {
        const uint64_t f = f0 + lane;
        const int route = f < H.n_frames ? frame_route(A, H, uint32_t(f)) : kRNone;
        const uint32_t sk = __ballot_sync(kFull, route == kRSkip);
        if (lane == 0 && sk) atomicAdd(&A.sc->skipped, (unsigned long long)__popc(sk));
        push_listed(A, route, kRDefer, uint32_t(f), lane, lt);
        push_listed(A, route, kRLane, uint32_t(f), lane, lt);
        push_listed(A, route, kRBig, uint32_t(f), lane, lt);
        push_listed(A, route, kRWarp, uint32_t(f), lane, lt);
    }
}

__global__ void __launch_bounds__(kAThreads, 2) apply_kernel(ApplyArgs A)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ASmem& S = *reinterpret_cast<ASmem*>(smem_raw);
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        int rc = check_header(A, &S.hdr);
        S.ok = rc == 0;
        if (rc) report(A.sc, rc);
        else if (blockIdx.x == 0) {
            A.sc->hdr_ok = 1;
            A.sc->target_version = S.hdr.target_v;
            A.sc->window = S.hdr.window;
            A.sc->n_frames = S.hdr.n_frames;
        }
    }
    __syncthreads();
    if (!S.ok) return;
    const Hdr H = S.hdr;
    const uint64_t V = H.target_v;
    AWarp& W = S.w[wid];
    // the frames route_kernel listed, or (self_route) every frame of the
    // stream, each checked, claimed and routed by lane 0 here
    const uint32_t nw = A.self_route ? 0u : min(A.sc->n_warp, A.defer_len);

    for (;;) {
        uint32_t j = 0;
        if (lane == 0) j = atomicAdd(&A.sc->frame_ticket, 1u);
        j = __shfl_sync(kFull, j, 0);
        uint32_t f = j;
        if (A.self_route) {
            if (j >= H.n_frames) break;
            int route = kRNone;
            if (lane == 0) {
                route = frame_route(A, H, j);
                if (route == kRSkip) atomicAdd(&A.sc->skipped, 1ull);
                else if (route == kRDefer) A.defer[atomicAdd(&A.sc->n_defer, 1u)] = j;
                else if (route == kRBig) A.defer[A.defer_len - 1 - atomicAdd(&A.sc->n_big, 1u)] = j;
            }
            if (__shfl_sync(kFull, route, 0) != kRWarp) continue;
        } else {
            if (j >= nw) break;
            f = A.warp[j];
        }
        const uint64_t fo = ld64(A.payload + H.idx_off + 8ull * f);
        const uint4 h0 = ld_nc16(A.payload + fo), h1 = ld_nc16(A.payload + fo + 16);
        const uint32_t kind = h0.y & 0xFFu;
        const uint32_t c = h0.z, raw = h0.w, bl = h1.x;
        const ChunkDesc cd = A.chunks[c];
        const bool is_xor = kind == kXorLz4 || kind == kXorRaw || kind == kXorSnappy;
        const bool cut = uint64_t(f) == A.abort_at;
        const uint32_t ub = cd.bits == 16 ? 2u : 1u;
        uint32_t lim = cut ? (A.split < raw ? A.split : raw) : raw;
        lim -= lim % ub;
        unsigned long long* st = &A.state[c];
        const Seg* ds = A.dst + cd.dst_begin;
        const uint8_t* body = A.payload + fo + kFrameHdr;
        bool good = true;
        if (kind == kXorRaw) {
            good = bl == raw;
            if (good) {
                for (uint32_t v = lane; v < raw / 16; v += 32) {
                    uint4 m = ld_nc16(body + 16 * v);
                    if (!is_zero(m)) xor_vec(A, cd, ds, 16 * v, m, lim);
                }
                for (uint32_t x = (raw & ~15u) + lane; x < raw; x += 32)
                    if (body[x] && x < lim) xor_byte(A.target, dst_of(ds, cd.dst_count, x), body[x]);
            }
        } else if (kind == kXorLz4) {
            for (uint32_t v = lane; v < bl / 16; v += 32)
                reinterpret_cast<uint4*>(W.body)[v] = ld_nc16(body + 16 * v);
            for (uint32_t x = (bl & ~15u) + lane; x < bl; x += 32) W.body[x] = body[x];
            __syncwarp();
            const int r = zsrc_apply<false>(A, cd, ds, W.body, bl, raw, lim, W, lane);
            __syncwarp();   // the body cache is reused by the next frame
            if (r == 2) {   // more non-zero bytes than the list holds (undone)
                if (lane == 0) A.defer[A.defer_len - 1 - atomicAdd(&A.sc->n_big, 1u)] = f;
                continue;
            }
            good = r == 1;
        } else if (kind == kOverwriteDense) {
            good = bl == raw;
            if (good) {
                for (uint32_t v = lane; v < raw / 16; v += 32)
                    put_vec(A, cd, ds, 16 * v, ld_nc16(body + 16 * v), lim, raw);
                for (uint32_t x = (raw & ~15u) + lane; x < raw; x += 32)
                    if (x < lim) A.target[dst_of(ds, cd.dst_count, x)] = body[x];
            }
        } else {
            // OVERWRITE records: n, ascending unit offsets, pad, values
            uint32_t cnt = bl >= 4 ? *reinterpret_cast<const uint32_t*>(body) : 0u;
            uint64_t pad = (4 - (2ull * cnt) % 4) % 4;
            good = bl >= 4 && 4 + 2ull * cnt + pad + uint64_t(cnt) * ub == bl;
            const uint16_t* offs = reinterpret_cast<const uint16_t*>(body + 4);
            const uint8_t* vals = body + 4 + 2 * cnt + pad;
            if (good) {
                bool bad = false;
                for (uint32_t i = lane; i < cnt; i += 32) {
                    uint32_t u = offs[i];
                    bad |= (u + 1) * ub > raw || (i && u <= offs[i - 1]);
                }
                good = !__any_sync(0xffffffffu, bad);
            }
            if (good) {
                for (uint32_t i = lane; i < cnt; i += 32) {
                    uint32_t x = uint32_t(offs[i]) * ub;
                    if (x >= lim) continue;
                    uint64_t a = dst_of(ds, cd.dst_count, x);
                    if (ub == 2 && (a & 1) == 0 && dst_of(ds, cd.dst_count, x + 1) == a + 1)
                        *reinterpret_cast<uint16_t*>(A.target + a) =
                            uint16_t(vals[2 * i] | (uint32_t(vals[2 * i + 1]) << 8));
                    else
                        for (uint32_t e = 0; e < ub; ++e)
                            A.target[dst_of(ds, cd.dst_count, x + e)] = vals[i * ub + e];
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            if (!good) {
                report(A.sc, DCR_ERR_CORRUPT);
            } else {
                atomicAdd(&A.sc->applied, 1ull);
                __threadfence();
                if (cut) {
                    A.sc->aborted = 1;
                    if (!is_xor) atomicExch(st, (V << 2) | kClaimed);
                } else {
                    atomicExch(st, (V << 2) | kDone);
                }
            }
        }
    }
}

// ---- small windows: one CTA per frame ------------------------------------
// apply_cta_kernel (256 threads): for windows with fewer frames than the GPU has warp
// slots, where one warp per frame would leave the run as long as one frame's
// serial token walk.  The CTA copies a ZSRC LZ4 body of up to kCBody bytes
// into shared memory, works out where a sequence starting at each body byte
// would end, builds 4- and 16-sequence jump tables by pointer doubling, and
// one thread follows the chain 16 sequences per step; the threads then
// expand the starts, decode one sequence each, place them by a prefix sum of
// their lengths, list the non-zero literal bytes in output order and check
// every match against that list (ZSRC: a match copies zero bytes only).
// Only a frame that passed every check is applied, its non-zero bytes XORed
// into the receiver spread evenly over the threads.  Other frames are
// applied CTA-wide (raw, overwrite, dense) or listed for the deferred
// kernels, as apply_kernel does.
constexpr int kCThreads = 256;
constexpr int kCWarps = kCThreads / 32;
constexpr uint32_t kCBody = 4096;               // body bytes walked in shared memory
constexpr uint32_t kCSeq = kCBody / 3 + 2;      // sequences such a body holds at most
constexpr uint16_t kCBad = 0xFFFF;              // no valid sequence starts here

struct __align__(16) CSmem {
    uint8_t body[kCBody + 16];
    uint16_t nxt[kCBody + 1];     // where the next sequence starts (n: the block ends here)
    uint16_t j4[kCBody + 1];      // ... four sequences on
    uint16_t j16[kCBody + 1];     // ... sixteen sequences on
    uint16_t start[kCSeq];        // every sequence's start
    uint16_t blk[kCSeq / 16 + 2]; // every sixteenth sequence's start
    uint32_t opos[kCSeq];         // output position of each sequence's literals
    uint16_t nz[kCBody];          // output positions of the non-zero literal bytes, ascending
    uint8_t nzv[kCBody];          // ... and their values
    unsigned long long wsum[kCWarps];
    Hdr hdr;
    uint32_t f, nseq;
    int ok;
};

// exclusive prefix sum of v over the CTA (two 32-bit counts packed in one
// 64-bit value); *total = the sum (every thread)
__device__ __forceinline__ unsigned long long cta_excl_scan(unsigned long long v, unsigned long long* wsum,
                                                            unsigned long long* total)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    unsigned long long incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long o = __shfl_up_sync(kFull, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    unsigned long long before = 0, tot = 0;
#pragma unroll
    for (int i = 0; i < kCWarps; ++i) {
        const unsigned long long x = wsum[i];
        before += i < w ? x : 0ull;
        tot += x;
    }
    __syncthreads();   // wsum is reused by the next scan
    *total = tot;
    return before + incl - v;
}

// The ZSRC LZ4 block body[0, n) (in S.body) applied to the chunk's receiver
// bytes below lim: 1 if applied, 0 if malformed or breaking the ZSRC promise
// (nothing written then).  Called by the whole CTA.
__device__ int zsrc_apply_cta(const ApplyArgs& A, const ChunkDesc& cd, const Seg* ds, uint32_t n, uint32_t raw,
                              uint32_t lim, CSmem& S)
{
    const int t = threadIdx.x;
    if (n == 0) return 0;   // an LZ4 block holds at least one token
    // where a sequence starting at each byte ends (n: the block's last
    // sequence; the end position n is absorbing)
    for (uint32_t p = t; p <= n; p += kCThreads) {
        uint16_t v = uint16_t(n);
        if (p < n) {
            const uint32_t e = seq_end(S.body, n, p);
            v = e == kEndBad ? kCBad : (e & kEndFinal) ? uint16_t(n) : e >= n ? kCBad : uint16_t(e);
        }
        S.nxt[p] = v;
    }
    __syncthreads();
    auto four = [&](const uint16_t* a, uint16_t* out) {   // out = a applied four times
        for (uint32_t p = t; p <= n; p += kCThreads) {
            uint16_t q = uint16_t(p);
#pragma unroll
            for (int r = 0; r < 4; ++r) q = q == kCBad ? kCBad : a[q];
            out[p] = q;
        }
        __syncthreads();
    };
    four(S.nxt, S.j4);
    four(S.j4, S.j16);
    if (t == 0) {   // the chain, sixteen sequences per step, then the last ones
        uint32_t p = 0, i = 0;
        bool bad = false;
        for (;;) {
            S.blk[i >> 4] = uint16_t(p);
            const uint16_t q = S.j16[p];
            if (q == kCBad || q == n) break;
            p = q;
            i += 16;
        }
        for (;;) {
            const uint16_t q = S.nxt[p];
            ++i;
            if (q == kCBad) { bad = true; break; }
            if (q == n) break;
            p = q;
        }
        S.nseq = bad ? 0u : i;
    }
    __syncthreads();
    const uint32_t nseq = S.nseq;
    if (nseq == 0) return 0;
    // every sequence's start, from the sixteenth before it
    for (uint32_t i = t; i < nseq; i += kCThreads) {
        uint32_t p = S.blk[i >> 4], r = i & 15;
        for (; r >= 4; r -= 4) p = S.j4[p];
        for (; r; --r) p = S.nxt[p];
        S.start[i] = uint16_t(p);
    }
    __syncthreads();
    // decode one sequence per thread (bytes bounds-checked by seq_end): place
    // them, check them, and list their non-zero literal bytes in order
    bool wrong = false;
    uint64_t carry = 0;
    uint32_t nzc = 0;
    for (uint32_t b0 = 0; b0 < nseq; b0 += kCThreads) {
        const uint32_t i = b0 + t;
        const bool mine = i < nseq, last = i + 1 == nseq;
        uint32_t q = 0, ll = 0, ml = 0, off = 0, lit = 0;
        if (mine) {
            q = S.start[i];
            const uint32_t tok = S.body[q++];
            ll = tok >> 4;
            if (ll == 15) {
                uint32_t b;
                do {
                    b = S.body[q++];
                    ll += b;
                } while (b == 255);
            }
            lit = q;
            q += ll;
            if (!last) {
                off = uint32_t(S.body[q]) | (uint32_t(S.body[q + 1]) << 8);
                q += 2;
                ml = tok & 15u;
                if (ml == 15) {
                    uint32_t b;
                    do {
                        b = S.body[q++];
                        ml += b;
                    } while (b == 255);
                }
                ml += 4;
            }
        }
        // the sequence's output length and its non-zero literal bytes,
        // scanned together (a length is below 2^21: at most 4096 literals, a
        // match of at most 19 + 255 bytes per body byte; 256 of them stay
        // below 2^32)
        uint32_t c = 0;
        if (mine)
            for (uint32_t k = 0; k < ll; ++k) c += S.body[lit + k] != 0;
        unsigned long long tot;
        const unsigned long long ex = cta_excl_scan(uint64_t(ll + ml) | (uint64_t(c) << 32), S.wsum, &tot);
        const uint64_t opl64 = carry + (ex & 0xFFFFFFFFull);
        const uint32_t opl = opl64 > raw ? raw + 1 : uint32_t(opl64);   // beyond the chunk: rejected below
        uint32_t at = nzc + uint32_t(ex >> 32);
        carry += tot & 0xFFFFFFFFull;
        nzc += uint32_t(tot >> 32);
        const uint32_t mop = opl + ll;
        if (mine) {
            S.opos[i] = opl;
            if (last) wrong |= opl > raw || ll != raw - opl;
            else wrong |= opl > raw || ll > raw - opl || off == 0 || off > mop || ml > raw - mop;
        }
        if (mine && !wrong)
            for (uint32_t k = 0; k < ll; ++k) {
                const uint8_t v = S.body[lit + k];
                if (v) {
                    S.nz[at] = uint16_t(opl + k);
                    S.nzv[at] = v;
                    ++at;
                }
            }
    }
    if (__syncthreads_or(wrong)) return 0;
    // every match copies [mop - off, + min(ml, off)) of the output: no listed
    // non-zero byte may fall there
    bool viol = false;
    for (uint32_t i = t; i + 1 < nseq; i += kCThreads) {
        uint32_t q = S.start[i];
        const uint32_t tok = S.body[q++];
        uint32_t ll = tok >> 4;
        if (ll == 15) {
            uint32_t b;
            do {
                b = S.body[q++];
                ll += b;
            } while (b == 255);
        }
        q += ll;
        const uint32_t off = uint32_t(S.body[q]) | (uint32_t(S.body[q + 1]) << 8);
        q += 2;
        uint32_t ml = tok & 15u;
        if (ml == 15) {
            uint32_t b;
            do {
                b = S.body[q++];
                ml += b;
            } while (b == 255);
        }
        ml += 4;
        const uint32_t s0 = S.opos[i] + ll - off, e0 = s0 + (ml < off ? ml : off);
        uint32_t lo = 0, hi = nzc;   // first listed position >= s0
        while (lo < hi) {
            const uint32_t mid = (lo + hi) >> 1;
            if (S.nz[mid] < s0) lo = mid + 1;
            else hi = mid;
        }
        viol |= lo < nzc && S.nz[lo] < e0;
    }
    if (__syncthreads_or(viol)) return 0;
    // the frame is valid: its non-zero bytes into the receiver
    const bool one = cd.dst_count == 1;
    const uint64_t base = one ? ds[0].addr - ds[0].off : 0ull;
    for (uint32_t j = t; j < nzc; j += kCThreads) {
        const uint32_t x = S.nz[j];
        if (x < lim) xor_byte(A.target, one ? base + x : dst_of(ds, cd.dst_count, x), S.nzv[j]);
    }
    return 1;
}

__global__ void __launch_bounds__(kCThreads) apply_cta_kernel(ApplyArgs A)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    CSmem& S = *reinterpret_cast<CSmem*>(smem_raw);
    const int t = threadIdx.x;
    if (t == 0) {
        const int rc = check_header(A, &S.hdr);
        S.ok = rc == 0;
        if (rc) report(A.sc, rc);
        else if (blockIdx.x == 0) {
            A.sc->hdr_ok = 1;
            A.sc->target_version = S.hdr.target_v;
            A.sc->window = S.hdr.window;
            A.sc->n_frames = S.hdr.n_frames;
        }
    }
    __syncthreads();
    if (!S.ok) return;
    const Hdr H = S.hdr;
    const uint64_t V = H.target_v;
    for (;;) {
        if (t == 0) S.f = atomicAdd(&A.sc->frame_ticket, 1u);
        __syncthreads();
        const uint32_t f = S.f;
        __syncthreads();
        if (f >= H.n_frames) break;
        // the frame's checks (every thread reads the same values)
        const uint64_t fo = ld64(A.payload + H.idx_off + 8ull * f);
        if (fo < kStreamHdr || fo % 16 || fo + kFrameHdr > H.idx_off) {
            if (t == 0) report(A.sc, DCR_ERR_CORRUPT);
            continue;
        }
        const uint4 h0 = ld_nc16(A.payload + fo), h1 = ld_nc16(A.payload + fo + 16);
        const uint32_t kind = h0.y & 0xFFu, fbits = (h0.y >> 8) & 0xFFu, fflags = h0.y >> 16;
        const uint32_t c = h0.z, raw = h0.w, bl = h1.x;
        if (h0.x != kFrameMagic || kind < kXorLz4 || kind > kXorSnappy || c < H.chunk_begin ||
            c >= H.chunk_begin + H.chunk_count || bl > H.idx_off - fo - kFrameHdr) {
            if (t == 0) report(A.sc, DCR_ERR_CORRUPT);
            continue;
        }
        const ChunkDesc cd = A.chunks[c];
        if (raw != cd.raw_len || fbits != cd.bits) {
            if (t == 0) report(A.sc, DCR_ERR_CORRUPT);
            continue;
        }
        const bool is_xor = kind == kXorLz4 || kind == kXorRaw || kind == kXorSnappy;
        if (A.retry_only && is_xor) {
            if (t == 0) report(A.sc, DCR_ERR_INVALID);
            continue;
        }
        if (uint64_t(f) > A.abort_at) continue;  // injected fault: never reached
        const bool cut = uint64_t(f) == A.abort_at;
        const uint32_t ub = cd.bits == 16 ? 2u : 1u;
        uint32_t lim = cut ? (A.split < raw ? A.split : raw) : raw;
        lim -= lim % ub;
        unsigned long long* st = &A.state[c];
        if (is_xor) {
            bool got = false;
            if (t == 0) {
                bool to = false;
                got = claim(st, V, &to);
                if (to) report(A.sc, DCR_ERR_TIMEOUT);
                if (!got && !to) atomicAdd(&A.sc->skipped, 1ull);
            }
            if (!__syncthreads_or(got)) continue;
            // Snappy frames and general LZ4 frames to the deferred kernels,
            // ZSRC LZ4 bodies larger than the shared buffer to big_kernel
            const bool zs = (fflags & kFrameZsrc) != 0;
            if (kind == kXorSnappy && zs) {
                if (t == 0) A.defer[A.defer_len - 1 - atomicAdd(&A.sc->n_big, 1u)] = f;
                continue;
            }
            if ((kind == kXorLz4 && !zs) || kind == kXorSnappy) {
                if (t == 0) A.defer[atomicAdd(&A.sc->n_defer, 1u)] = f;
                continue;
            }
            if (kind == kXorLz4 && bl > kCBody) {
                if (t == 0) A.defer[A.defer_len - 1 - atomicAdd(&A.sc->n_big, 1u)] = f;
                continue;
            }
        }
        const Seg* ds = A.dst + cd.dst_begin;
        const uint8_t* body = A.payload + fo + kFrameHdr;
        bool good = true;
        if (kind == kXorRaw) {
            good = bl == raw;
            if (good) {
                for (uint32_t v = t; v < raw / 16; v += kCThreads) {
                    const uint4 m = ld_nc16(body + 16 * v);
                    if (!is_zero(m)) xor_vec(A, cd, ds, 16 * v, m, lim);
                }
                for (uint32_t x = (raw & ~15u) + t; x < raw; x += kCThreads)
                    if (body[x] && x < lim) xor_byte(A.target, dst_of(ds, cd.dst_count, x), body[x]);
            }
        } else if (kind == kXorLz4) {
            for (uint32_t v = t; v < bl / 16; v += kCThreads)
                reinterpret_cast<uint4*>(S.body)[v] = ld_nc16(body + 16 * v);
            for (uint32_t x = (bl & ~15u) + t; x < bl; x += kCThreads) S.body[x] = body[x];
            __syncthreads();
            good = zsrc_apply_cta(A, cd, ds, bl, raw, lim, S) == 1;
        } else if (kind == kOverwriteDense) {
            good = bl == raw;
            if (good) {
                for (uint32_t v = t; v < raw / 16; v += kCThreads)
                    put_vec(A, cd, ds, 16 * v, ld_nc16(body + 16 * v), lim, raw);
                for (uint32_t x = (raw & ~15u) + t; x < raw; x += kCThreads)
                    if (x < lim) A.target[dst_of(ds, cd.dst_count, x)] = body[x];
            }
        } else {
            // OVERWRITE records: n, ascending unit offsets, pad, values
            const uint32_t cnt = bl >= 4 ? *reinterpret_cast<const uint32_t*>(body) : 0u;
            const uint64_t pad = (4 - (2ull * cnt) % 4) % 4;
            good = bl >= 4 && 4 + 2ull * cnt + pad + uint64_t(cnt) * ub == bl;
            const uint16_t* offs = reinterpret_cast<const uint16_t*>(body + 4);
            const uint8_t* vals = body + 4 + 2 * cnt + pad;
            if (good) {
                bool bad = false;
                for (uint32_t i = t; i < cnt; i += kCThreads) {
                    const uint32_t u = offs[i];
                    bad |= (u + 1) * ub > raw || (i && u <= offs[i - 1]);
                }
                good = !__syncthreads_or(bad);
            }
            if (good) {
                for (uint32_t i = t; i < cnt; i += kCThreads) {
                    const uint32_t x = uint32_t(offs[i]) * ub;
                    if (x >= lim) continue;
                    const uint64_t a = dst_of(ds, cd.dst_count, x);
                    if (ub == 2 && (a & 1) == 0 && dst_of(ds, cd.dst_count, x + 1) == a + 1)
                        *reinterpret_cast<uint16_t*>(A.target + a) =
                            uint16_t(vals[2 * i] | (uint32_t(vals[2 * i + 1]) << 8));
                    else
                        for (uint32_t e = 0; e < ub; ++e)
                            A.target[dst_of(ds, cd.dst_count, x + e)] = vals[i * ub + e];
                }
            }
        }
        __syncthreads();   // every thread's writes of this frame precede its DONE mark
        if (t == 0) {
            if (!good) {
                report(A.sc, DCR_ERR_CORRUPT);
            } else {
                atomicAdd(&A.sc->applied, 1ull);
                __threadfence();
                if (cut) {
                    A.sc->aborted = 1;
                    if (!is_xor) atomicExch(st, (V << 2) | kClaimed);
                } else {
                    atomicExch(st, (V << 2) | kDone);
                }
            }
        }
    }
}

// General LZ4 frames (no ZSRC promise): full decode in shared memory.
__global__ void __launch_bounds__(kDThreads) defer_kernel(ApplyArgs A)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    uint8_t* out = smem_raw;                       // kChunk bytes
    __shared__ uint32_t s_f, s_good;
    // final: the first phase (route, apply or CTA kernel) lists deferred frames
    if (!A.sc->hdr_ok || *reinterpret_cast<volatile uint32_t*>(&A.sc->n_defer) == 0) return;
    const uint8_t* p = A.payload;
    const uint64_t total = ld64(p + 56), nf = ld64(p + 48), idx_off = total - 8 * nf;
    const uint64_t V = ld64(p + 24);
    const int lane = threadIdx.x & 31;
    for (;;) {
        if (threadIdx.x == 0) {
            uint32_t j = atomicAdd(&A.sc->defer_ticket, 1u);
            s_f = j < *reinterpret_cast<volatile uint32_t*>(&A.sc->n_defer) ? A.defer[j] : UINT32_MAX;
        }
        __syncthreads();
        const uint32_t f = s_f;
        if (f == UINT32_MAX) break;
        const uint64_t fo = ld64(p + idx_off + 8ull * f);
        const uint4 h0 = ld_nc16(p + fo), h1 = ld_nc16(p + fo + 16);
        const uint32_t c = h0.z, raw = h0.w, n = h1.x;
        const bool zs = ((h0.y >> 16) & kFrameZsrc) != 0;   // matches must copy zeros
        const bool snappy = (h0.y & 0xFFu) == kXorSnappy;
        const ChunkDesc cd = A.chunks[c];
        const bool cut = uint64_t(f) == A.abort_at;
        const uint32_t ub = cd.bits == 16 ? 2u : 1u;
        uint32_t lim = cut ? (A.split < raw ? A.split : raw) : raw;
        lim -= lim % ub;
        const uint8_t* src = p + fo + kFrameHdr;
        if (threadIdx.x < 32) {
            const bool good = snappy ? warp_decode_snappy(src, n, out, raw, zs, lane)
                                     : warp_decode_lz4(src, n, out, raw, zs, lane);
            if (lane == 0) s_good = good;
        }
        __syncthreads();
        if (s_good) {
            const Seg* ds = A.dst + cd.dst_begin;
            for (uint32_t v = threadIdx.x; v < raw / 16; v += kDThreads) {
                uint4 m = reinterpret_cast<const uint4*>(out)[v];
                if (!is_zero(m)) xor_vec(A, cd, ds, 16 * v, m, lim);
            }
            for (uint32_t x = (raw & ~15u) + threadIdx.x; x < raw; x += kDThreads)
                if (out[x] && x < lim) xor_byte(A.target, dst_of(ds, cd.dst_count, x), out[x]);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            if (!s_good) {
                report(A.sc, DCR_ERR_CORRUPT);
            } else {
                atomicAdd(&A.sc->applied, 1ull);
                __threadfence();
                if (cut) A.sc->aborted = 1;
                else atomicExch(&A.state[c], (V << 2) | kDone);
            }
        }
        __syncthreads();
    }
}

// Large ZSRC frames (body beyond the cache, or more non-zero bytes than the
// list holds): one warp per frame, body read from global memory, matches
// checked against a bitmap of the non-zero output bytes.  The frames were
// validated and claimed by apply_kernel.
template <class WS>
__global__ void __launch_bounds__(32 * WS::kWarps, 3) big_kernel(ApplyArgs A)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    WS& W = reinterpret_cast<WS*>(smem_raw)[threadIdx.x >> 5];
    const int lane = threadIdx.x & 31;
    if (!A.sc->hdr_ok) return;
    const uint8_t* p = A.payload;
    const uint64_t total = ld64(p + 56), nf = ld64(p + 48), idx_off = total - 8 * nf;
    const uint64_t V = ld64(p + 24);
    const uint32_t nbig = A.sc->n_big;   // final: written by the first phase (route, apply, CTA and lane kernels)
    if (nbig == 0) return;
    for (;;) {
        uint32_t j = 0;
        if (lane == 0) j = atomicAdd(&A.sc->big_ticket, 1u);
        j = __shfl_sync(kFull, j, 0);
        if (j >= nbig) break;
        const uint32_t f = A.defer[A.defer_len - 1 - j];
        const uint64_t fo = ld64(p + idx_off + 8ull * f);
        const uint4 h0 = ld_nc16(p + fo), h1 = ld_nc16(p + fo + 16);
        const bool sn = (h0.y & 0xFFu) == kXorSnappy;   // ZSRC Snappy frames walk the same way
        const uint32_t c = h0.z, raw = h0.w, bl = h1.x;
        const ChunkDesc cd = A.chunks[c];
        const bool cut = uint64_t(f) == A.abort_at;
        const uint32_t ub = cd.bits == 16 ? 2u : 1u;
        uint32_t lim = cut ? (A.split < raw ? A.split : raw) : raw;
        lim -= lim % ub;
        const uint8_t* body = p + fo + kFrameHdr;
        const Seg* ds = A.dst + cd.dst_begin;
        int r = 0;
        if (WS::kSplit && bl <= kSBody) {
            if constexpr (WS::kSplit) {
                // the body into shared memory: whole vectors, then the bytes after them
                const uint32_t nv = bl / 16;
                for (uint32_t v = lane; v < nv; v += 32)
                    reinterpret_cast<uint4*>(W.body)[v] = ld_nc16(body + 16 * v);
                for (uint32_t i = 16 * nv + lane; i < bl; i += 32) W.body[i] = body[i];
                __syncwarp();
                r = sn ? split_apply<SnappyWalk>(A, cd, ds, W.body, bl, raw, lim, W, lane)
                       : split_apply<Lz4Walk>(A, cd, ds, W.body, bl, raw, lim, W, lane);
            }
        } else {
            r = sn ? zsrc_apply<true, WS, SnappyWalk>(A, cd, ds, body, bl, raw, lim, W, lane)
                   : zsrc_apply<true, WS>(A, cd, ds, body, bl, raw, lim, W, lane);
        }
        __syncwarp();   // the bitmap is reused by the next frame
        if (lane == 0) {
            if (r != 1) {
                report(A.sc, DCR_ERR_CORRUPT);
            } else {
                atomicAdd(&A.sc->applied, 1ull);
                __threadfence();
                if (cut) A.sc->aborted = 1;
                else atomicExch(&A.state[c], (V << 2) | kDone);
            }
        }
    }
}

// ---- ZSRC frames, one thread each -----------------------------------------
// In a ZSRC block every match (LZ4) or copy (Snappy) copies zero bytes, so
// the non-zero output bytes are literal bytes.  lane_kernel gives each frame
// one thread, which walks the block in order as a serial decoder would but
// writes only the non-zero literal bytes (XORed into the receiver, combined
// per 32-bit word).  Of the output so far it keeps a few zero stretches:
// every byte from z1 on (one past the last non-zero byte), the bytes [g0, g1)
// between the last two non-zero bytes, and the longest zero runs the
// library's encoder copies from (LaneOut).  A match whose source lies inside
// one of them provably copies zeros.  For one that does not, and for a malformed
// block, the thread undoes what it XORed (XOR is self-inverse) and passes the
// frame to big_kernel, whose bitmap check over the whole output decides.
// Per element this costs a few dozen instructions of one thread, against a
// warp's worth in the cooperative walks, which pays when a window has many
// frames.
constexpr int kLThreads = 128;

#include "lane.cuh"

// Receiver address of canonical chunk offset x, for x that never decreases.
struct LaneDst {
    const Seg* s;
    uint32_t n, i, next;
    uint64_t base;
    __device__ __forceinline__ void init(const Seg* ds, uint32_t cnt)
    {
        s = ds;
        n = cnt;
        i = 0;
        base = s[0].addr - s[0].off;
        next = n > 1 ? s[1].off : 0xFFFFFFFFu;
    }
    __device__ __forceinline__ uint64_t addr(uint32_t x)
    {
        while (x >= next) {
            ++i;
            base = s[i].addr - s[i].off;
            next = i + 1 < n ? s[i + 1].off : 0xFFFFFFFFu;
        }
        return base + x;
    }
};

// XOR bytes into the receiver, one reduction per 32-bit word touched in a row.
struct LaneXor {
    uint8_t* t;
    uint64_t wa;
    uint32_t wv;
    __device__ __forceinline__ void flush()
    {
        if (wv) asm volatile("red.global.xor.b32 [%0], %1;" ::"l"(t + wa), "r"(wv) : "memory");
        wv = 0;
    }
    __device__ __forceinline__ void add(uint64_t a, uint32_t b)
    {
        const uint64_t w = a & ~3ull;   // the arena is 16-byte aligned
        if (w != wa) {
            flush();
            wa = w;
        }
        wv ^= b << (8 * (a & 3));
    }
};

// lane_kernel's sink: non-zero literal bytes below lim XORed into the
// receiver through the chunk's pieces.
struct ApplySink {
    LaneDst D;
    LaneXor X;
    uint32_t lim;
    __device__ __forceinline__ void lit(uint32_t x, uint32_t b)
    {
        if (x < lim) X.add(D.addr(x), b);
    }
};

__global__ void __launch_bounds__(kLThreads, 7) lane_kernel(ApplyArgs A)
{
    if (!A.sc->hdr_ok) return;
    const uint32_t nl = A.sc->n_lane;   // final: written by route_kernel
    if (nl == 0) return;
    const uint8_t* p = A.payload;
    const uint64_t total = ld64(p + 56), nf = ld64(p + 48), idx_off = total - 8 * nf;
    const uint64_t V = ld64(p + 24);
    const int lane = threadIdx.x & 31;
    // 32 consecutive list entries per warp, spread over the blocks first
    const uint32_t wpb = kLThreads / 32, nw = gridDim.x * wpb;
    uint32_t applied = 0;
    for (uint32_t g = (threadIdx.x >> 5) * gridDim.x + blockIdx.x; 32ull * g < nl; g += nw) {
        const uint32_t j = 32 * g + lane;
        const bool mine = j < nl;
        LaneWalk<ApplySink> W;
        uint32_t f = 0, c = 0;
        bool cut = false, act = false;
        int res = kLStop;
        const uint8_t* body = nullptr;
        const Seg* ds = nullptr;
        uint32_t dcnt = 1;
        if (mine) {
            f = A.lane[j];
            const uint64_t fo = ld64(p + idx_off + 8ull * f);
            const uint4 h0 = ld_nc16(p + fo), h1 = ld_nc16(p + fo + 16);
            const uint32_t raw = h0.w;
            c = h0.z;
            const ChunkDesc cd = A.chunks[c];
            cut = uint64_t(f) == A.abort_at;
            const uint32_t ub = cd.bits == 16 ? 2u : 1u;
            uint32_t lim = cut ? (A.split < raw ? A.split : raw) : raw;
            lim -= lim % ub;
            body = p + fo + kFrameHdr;
            ds = A.dst + cd.dst_begin;
            dcnt = cd.dst_count;
            W.init((h0.y & 0xFFu) == kXorSnappy, body, h1.x, raw, 0);
            W.K.D.init(ds, dcnt);
            W.K.X = LaneXor{A.target, ~0ull, 0u};
            W.K.lim = lim;
            act = !W.sn || snappy_pre(W);
        }
        lane_run<false>(W, act, res);
        if (mine) W.K.X.flush();
        const bool ok = mine && res == kLValid;
        if (ok) {
            ++applied;
            __threadfence();
            if (cut) A.sc->aborted = 1;
            else atomicExch(&A.state[c], (V << 2) | kDone);
        }
        // a frame that is not proven: XOR its literals again (the bytes below
        // the first walk's `done`), then big_kernel decides
        const bool undo = mine && !ok && W.O.done > 0;
        if (__any_sync(kFull, undo)) {
            bool act2 = false;
            if (undo) {
                W.init(W.sn, body, W.n, W.raw, W.O.done);
                W.K.D.init(ds, dcnt);
                W.K.X = LaneXor{A.target, ~0ull, 0u};
                act2 = !W.sn || snappy_pre(W);
            }
            int r2 = kLStop;
            lane_run<true>(W, act2, r2);
            if (undo) W.K.X.flush();
        }
        if (mine && !ok) A.defer[A.defer_len - 1 - atomicAdd(&A.sc->n_big, 1u)] = f;
    }
    applied = __reduce_add_sync(kFull, applied);
    if (lane == 0 && applied) atomicAdd(&A.sc->applied, (unsigned long long)applied);
}

// Commit rule: every chunk with a frame in the stream is DONE for the target.
__global__ void pending_kernel(ApplyArgs A)
{
    if (!A.sc->hdr_ok) return;
    const uint8_t* p = A.payload;
    const uint64_t total = ld64(p + 56), nf = ld64(p + 48), idx_off = total - 8 * nf;
    const uint64_t V = ld64(p + 24);
    const uint32_t cb = *reinterpret_cast<const uint32_t*>(p + 40);
    const uint32_t cc = *reinterpret_cast<const uint32_t*>(p + 44);
    unsigned long long pend = 0;
    for (uint64_t f = blockIdx.x * uint64_t(blockDim.x) + threadIdx.x; f < nf;
         f += uint64_t(gridDim.x) * blockDim.x) {
        uint64_t fo = ld64(p + idx_off + 8 * f);
        if (fo < kStreamHdr || fo % 16 || fo + kFrameHdr > idx_off) { ++pend; continue; }
        uint32_t c = *reinterpret_cast<const uint32_t*>(p + fo + 8);
        if (c < cb || c >= cb + cc) { ++pend; continue; }
        if (*reinterpret_cast<volatile unsigned long long*>(&A.state[c]) != ((V << 2) | kDone)) ++pend;
    }
    pend = __reduce_add_sync(0xffffffffu, unsigned(pend));
    if ((threadIdx.x & 31) == 0 && pend) atomicAdd(&A.sc->pending, pend);
}

}  // namespace

int apply_kernel_config(KernelConfig* kc)
{
    cudaError_t e = cudaFuncSetAttribute(apply_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(sizeof(ASmem)));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(defer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kChunk));
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&kc->apply_blocks_per_sm, apply_kernel, kAThreads,
                                                          sizeof(ASmem));
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&kc->defer_blocks_per_sm, defer_kernel, kDThreads,
                                                          kChunk);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(big_kernel<BWarp>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(sizeof(BWarp) * BWarp::kWarps));
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&kc->big_blocks_per_sm, big_kernel<BWarp>,
                                                          32 * BWarp::kWarps, sizeof(BWarp) * BWarp::kWarps);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(big_kernel<SWarp>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(sizeof(SWarp) * SWarp::kWarps));
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&kc->split_blocks_per_sm, big_kernel<SWarp>,
                                                          32 * SWarp::kWarps, sizeof(SWarp) * SWarp::kWarps);
    if (e == cudaSuccess)   // no shared memory: all of it as L1 for the bodies
        e = cudaFuncSetAttribute(lane_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 0);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&kc->lane_blocks_per_sm, lane_kernel, kLThreads, 0);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(apply_cta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sizeof(CSmem)));
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&kc->apply_cta_blocks_per_sm, apply_cta_kernel, kCThreads,
                                                          sizeof(CSmem));
    if (e == cudaSuccess) {
        // load the kernels of the apply that no query above touched, so that
        // no apply call loads code lazily
        cudaFuncAttributes fa;
        e = cudaFuncGetAttributes(&fa, pending_kernel);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, route_kernel);
    }
    if (e != cudaSuccess) return cuda_error(e, "apply kernel configuration");
    if (kc->apply_blocks_per_sm < 1) kc->apply_blocks_per_sm = 1;
    if (kc->apply_cta_blocks_per_sm < 1) kc->apply_cta_blocks_per_sm = 1;
    if (kc->big_blocks_per_sm < 1) kc->big_blocks_per_sm = 1;
    if (kc->split_blocks_per_sm < 1) kc->split_blocks_per_sm = 1;
    if (kc->lane_blocks_per_sm < 1) kc->lane_blocks_per_sm = 1;
    if (kc->defer_blocks_per_sm < 1) kc->defer_blocks_per_sm = 1;
    return DCR_OK;
}

namespace {

// The first phase of an apply: one CTA per frame for plans whose windows
// have fewer chunks than the GPU has warp slots (or when the plan asks for
// it), else route_kernel and one warp per frame; then lane_kernel for the
// ZSRC frames routed to it.  Returns the kernels launched.
int launch_first(const dcr_plan* P, const ApplyArgs& A, cudaStream_t s)
{
    const int sms = P->kc.num_sms;
    const bool cta = P->apply == DCR_APPLY_CTA ||
                     (P->apply == DCR_APPLY_AUTO && P->max_window_chunks <= uint64_t(P->small_window_chunks));
    if (cta) {   // lists nothing for lane_kernel
        apply_cta_kernel<<<sms * P->kc.apply_cta_blocks_per_sm, kCThreads, sizeof(CSmem), s>>>(A);
        return 1;
    }
    if (A.self_route) {   // no stream of this plan reaches lane_kernel
        apply_kernel<<<sms * P->kc.apply_blocks_per_sm, kAThreads, sizeof(ASmem), s>>>(A);
        return 1;
    }
    route_kernel<<<sms * 4, kRtThreads, 0, s>>>(A);
    apply_kernel<<<sms * P->kc.apply_blocks_per_sm, kAThreads, sizeof(ASmem), s>>>(A);
    lane_kernel<<<sms * P->kc.lane_blocks_per_sm, kLThreads, 0, s>>>(A);
    return 3;
}

}  // namespace

namespace {

// Frames in a stream from which its ZSRC frames go to lane_kernel.
// lane_kernel spends a third of apply_kernel's instructions per frame (a
// tenth of big_kernel's) but walks a frame several times slower: one
// thread's chain of a few hundred instructions per sequence.  Its run lasts
// at least one frame's walk, which the warp kernels' whole run undercuts
// until the stream fills about a quarter of lane_kernel's thread slots
// (measured: 16 384 frames of 1 % masks, 0.65 ms in lane_kernel against
// 0.28 ms in apply_kernel; 131 072, 1.4-1.8 against 2.2 ms).
uint64_t lane_min_frames(const dcr_plan* P)
{
    if (P->apply == DCR_APPLY_LANE) return 0;
    const uint64_t t = uint64_t(P->kc.num_sms) * P->kc.lane_blocks_per_sm * kLThreads / 4;
    // launch_first leaves lane_kernel out for plans whose windows are smaller
    return P->apply == DCR_APPLY_WARP || P->apply == DCR_APPLY_SPLIT || P->max_window_chunks < t ? UINT64_MAX : t;
}

ApplyArgs make_args(const dcr_plan* P, dcr_recv_state* st, const void* payload, size_t size, void* target,
                    uint64_t abort_at, uint32_t split, int retry_only)
{
    ApplyArgs A{};
    A.chunks = P->d_chunks;
    A.dst = P->d_dst;
    A.win = P->d_win;
    A.n_windows = uint32_t(P->win_start.size() - 1);
    A.retry_only = retry_only;
    A.payload = static_cast<const uint8_t*>(payload);
    A.size = size;
    A.target = static_cast<uint8_t*>(target);
    A.state = reinterpret_cast<unsigned long long*>(st->d_chunk_state);
    A.sc = st->d_scratch;
    A.defer = st->d_defer;
    A.lane = st->d_defer + (P->max_window_chunks + 1);
    A.warp = st->d_defer + 2 * (P->max_window_chunks + 1);
    A.lane_min = lane_min_frames(P);
    A.self_route = A.lane_min == UINT64_MAX;
    A.split_all = P->apply == DCR_APPLY_SPLIT;
    A.defer_len = uint32_t(P->max_window_chunks + 1);
    A.plan_hash = P->hash;
    A.version = st->version;
    A.abort_at = abort_at;
    A.split = split;
    return A;
}

// the kernels of the frames the first phase deferred: general LZ4 and
// Snappy frames; the ZSRC frames that lane_kernel could not prove, and those
// the first kernels pass on, for big_kernel
void launch_deferred(const dcr_plan* P, const ApplyArgs& A, cudaStream_t s)
{
    const int sms = P->kc.num_sms;
    defer_kernel<<<sms * P->kc.defer_blocks_per_sm, kDThreads, kChunk, s>>>(A);
    if (P->codec == DCR_CODEC_SNAPPY || P->apply == DCR_APPLY_SPLIT)
        big_kernel<SWarp><<<sms * P->kc.split_blocks_per_sm, 32 * SWarp::kWarps, sizeof(SWarp) * SWarp::kWarps, s>>>(A);
    else
        big_kernel<BWarp><<<sms * P->kc.big_blocks_per_sm, 32 * BWarp::kWarps, sizeof(BWarp) * BWarp::kWarps, s>>>(A);
}

}  // namespace

int apply_launch_part(const dcr_plan* P, dcr_recv_state* st, const void* payload, size_t size, void* target,
                      uint64_t abort_at, uint32_t split, int retry_only, int part, cudaStream_t s)
{
    const ApplyArgs A = make_args(P, st, payload, size, target, abort_at, split, retry_only);
    cudaError_t e = cudaSuccess;
    const int sms = P->kc.num_sms;
    if (part != kApplyDeferred) {
        e = cudaMemsetAsync(st->d_scratch, 0, sizeof(ApplyScratch), s);
        if (e != cudaSuccess) return cuda_error(e, "apply scratch reset");
        if (P->profiling) cudaEventRecord(P->ev[3], s);
        P->apply_kernels = uint32_t(launch_first(P, A, s)) + 1;   // and the commit check
        if (P->profiling) cudaEventRecord(P->ev[4], s);
    }
    if (part != kApplyFirst) {
        if (part == kApplyDeferred) {   // the commit check runs again after them
            e = cudaMemsetAsync(&st->d_scratch->pending, 0, sizeof(st->d_scratch->pending), s);
            if (e != cudaSuccess) return cuda_error(e, "apply scratch reset");
            if (P->profiling) cudaEventRecord(P->ev[7], s);
        }
        launch_deferred(P, A, s);
        P->apply_kernels += part == kApplyDeferred ? 3 : 2;
    }
    if (P->profiling) cudaEventRecord(P->ev[5], s);
    pending_kernel<<<sms, 256, 0, s>>>(A);
    if (P->profiling) cudaEventRecord(P->ev[6], s);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "apply launch");
    return DCR_OK;
}

int apply_launch(const dcr_plan* P, dcr_recv_state* st, const void* payload, size_t size, void* target,
                 uint64_t abort_at, uint32_t split, int retry_only, cudaStream_t s)
{
    return apply_launch_part(P, st, payload, size, target, abort_at, split, retry_only, kApplyAll, s);
}

// ---- apply without allocation ---------------------------------------------
// dcr_apply_noalloc runs the same three kernels as dcr_apply, but the call's
// scratch (the ApplyScratch counters and the list of deferred frames) lives
// in the file-scope device array below instead of the receiver state's
// buffers.  Its callers cannot allocate device memory when a refit arrives:
// an inference engine typically reserves nearly all free HBM for its KV cache
// at start-up and runs the weight update from a hook where a cudaMalloc (or
// PyTorch's caching allocator growing its pool) would fail or stall serving.
// The call itself neither allocates nor frees device or pinned memory; the
// status comes back through a stack buffer.
namespace {

constexpr uint32_t kNoallocMaxChunks = 65536;    // window limit: 4 GiB of canonical bytes
constexpr size_t kNoallocHead = 256;             // ApplyScratch, padded
static_assert(sizeof(ApplyScratch) <= kNoallocHead, "counters fit the head");
constexpr size_t kNoallocBytes = kNoallocHead + 12 * (size_t(kNoallocMaxChunks) + 1);   // 768 KiB + 268 B

// [0, 256): ApplyScratch, cleared by a memset on the caller's stream at the
// start of every call; [256, ...): deferred frame list, written before read.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
struct NoallocAddr {
    unsigned long long ctx;   // unique id of the context the address belongs to (0: unknown)
    void* ptr;
};
NoallocAddr g_noalloc[kMaxDevices] = {};

// Unique id of the calling thread's current CUDA context, or 0 if the
// driver cannot tell.  The two driver calls are looked up through the
// runtime, so the library does not link the driver library itself.
unsigned long long current_ctx_id()
{
    using GetCur = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCur get_cur = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_cur = reinterpret_cast<GetCur>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetId>(f);
    });
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (!get_cur || !get_id || get_cur(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of this device's copy of the array, looked up with that
// device current and kept with the id of the context it was found in: a
// new context (after cudaDeviceReset, or a released primary context) gets
// the address looked up again instead of a stale one.  The lookup may load
// the module, which allocates; dcr_recv_state_create does it once so that
// dcr_apply_noalloc itself does not.
int noalloc_scratch(int dev, void** out)
{
    if (dev < 0 || dev >= kMaxDevices) return set_error(DCR_ERR_INVALID, "device %d out of range", dev);
    const unsigned long long ctx = current_ctx_id();
    std::lock_guard<std::mutex> g(g_noalloc_mu);
    NoallocAddr& a = g_noalloc[dev];
    if (!a.ptr || ctx == 0 || a.ctx != ctx) {
        void* ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_error(e, "cudaGetSymbolAddress of the static apply scratch");
        a.ptr = ptr;
        a.ctx = ctx;
    }
    *out = a.ptr;
    return DCR_OK;
}

}  // namespace

int noalloc_prepare()
{
    int dev = -1;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    void* ptr = nullptr;
    return noalloc_scratch(dev, &ptr);
}

int apply_launch_noalloc(const dcr_plan* P, dcr_recv_state* st, const void* payload, size_t size,
                         void* target, ApplyScratch** sc_out, cudaStream_t s)
{
    if (P->max_window_chunks > kNoallocMaxChunks)
        return set_error(DCR_ERR_CAPACITY,
                         "dcr_apply_noalloc: windows of %llu chunks exceed the static scratch limit of %u "
                         "chunks (build the plan with window_bytes <= 4 GiB)",
                         (unsigned long long)P->max_window_chunks, kNoallocMaxChunks);
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (dev != P->device) return set_error(DCR_ERR_INVALID, "dcr_apply_noalloc: plan belongs to device %d", P->device);
    void* base = nullptr;
    int rc = noalloc_scratch(dev, &base);
    if (rc) return rc;
    ApplyArgs A{};
    A.chunks = P->d_chunks;
    A.dst = P->d_dst;
    A.win = P->d_win;
    A.n_windows = uint32_t(P->win_start.size() - 1);
    A.retry_only = 0;
    A.payload = static_cast<const uint8_t*>(payload);
    A.size = size;
    A.target = static_cast<uint8_t*>(target);
    A.state = reinterpret_cast<unsigned long long*>(st->d_chunk_state);
    A.sc = static_cast<ApplyScratch*>(base);
    A.defer = reinterpret_cast<uint32_t*>(static_cast<unsigned char*>(base) + kNoallocHead);
    A.defer_len = kNoallocMaxChunks + 1;
    A.lane = A.defer + A.defer_len;
    A.warp = A.defer + 2 * A.defer_len;
    A.lane_min = lane_min_frames(P);
    A.self_route = A.lane_min == UINT64_MAX;
    A.split_all = P->apply == DCR_APPLY_SPLIT;
    A.plan_hash = P->hash;
    A.version = st->version;
    A.abort_at = DCR_NO_FAULT;
    A.split = 0;
    e = cudaMemsetAsync(A.sc, 0, sizeof(ApplyScratch), s);
    if (e != cudaSuccess) return cuda_error(e, "static apply scratch reset");
    const int sms = P->kc.num_sms;
    launch_first(P, A, s);
    launch_deferred(P, A, s);
    pending_kernel<<<sms, 256, 0, s>>>(A);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "apply launch");
    *sc_out = A.sc;
    return DCR_OK;
}

}  // namespace dcr

extern "C" int dcr_apply_noalloc(const dcr_plan* p, dcr_recv_state* st, const void* payload, size_t size,
                                 void* target, dcr_apply_result* result, void* stream)
{
    using namespace dcr;
    if (result) memset(result, 0, sizeof(*result));
    if (!p || !st || !payload || !target) return set_error(DCR_ERR_INVALID, "dcr_apply_noalloc: NULL argument");
    if (st->plan != p) return set_error(DCR_ERR_INVALID, "dcr_apply_noalloc: state belongs to another plan");
    if (size < kStreamHdr) return set_error(DCR_ERR_CORRUPT, "dcr_apply_noalloc: stream shorter than its header");
    if ((reinterpret_cast<uintptr_t>(payload) | reinterpret_cast<uintptr_t>(target)) & 15)
        return set_error(DCR_ERR_INVALID, "dcr_apply_noalloc: payload/target not 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ApplyScratch* dsc = nullptr;
    int rc = apply_launch_noalloc(p, st, payload, size, target, &dsc, s);
    if (rc) return rc;
    ApplyScratch a;   // pageable stack copy of the counters
    cudaError_t e = cudaMemcpyAsync(&a, dsc, sizeof(a), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_error(e, "dcr_apply_noalloc status read");
    if (result) {
        result->target_version = a.target_version;
        result->n_frames = a.n_frames;
        result->frames_applied = a.applied;
        result->frames_skipped = a.skipped;
        result->pending = a.pending;
        result->window = a.window;
    }
    if (a.err) return set_error(a.err, "dcr_apply_noalloc: device reported error %d", a.err);
    if (a.pending)
        return set_error(DCR_ERR_INCOMPLETE, "dcr_apply_noalloc: %llu framed chunks not done",
                         (unsigned long long)a.pending);
    // commit rule of dcr_apply: the version advances once every window of the
    // target version has been applied
    if (a.target_version != st->pending) {
        std::fill(st->win_done.begin(), st->win_done.end(), 0);
        st->pending = a.target_version;
    }
    st->win_done[a.window] = 1;
    bool all = true;
    for (uint8_t d : st->win_done) all = all && d;
    if (all) {
        st->version = a.target_version;
        st->pending = ~0ull;
        if (result) result->committed = 1;
    }
    return DCR_OK;
}
