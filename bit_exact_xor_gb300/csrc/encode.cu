// Sender hot path: one persistent, warp-specialised kernel per window.
//
// Per 64 KiB canonical chunk it gathers old and new through the plan's
// shard->canonical pieces, forms mask = old XOR new in shared memory, counts
// changed stored values, encodes the chunk (LZ4 block, raw mask, overwrite
// records or dense overwrite) and writes the frame straight to its final
// place in the stream, found by a decoupled look-back over the frame sizes
// of earlier chunks.  A small second kernel writes the frame index and the
// stream header.
//
// Method: "GPU-accelerated weight teleportation", "Delta update algebra"
// (mask = old XOR new on raw bits) and "A strong baseline with the
// Blackwell-native DE" (LZ4 block format); NeMo-DCR paper summary, "Input and
// change detection" (bitwise compare per owner shard), "Direct Projection",
// "Residual Conversion" and "Hybrid encoding and compression" (XOR masks for
// affine changes, overwrites for residual ones).
//
// Structure.  One CTA per SM: 16 loader warps and 2 encoder warps share two
// chunk buffers in shared memory.  Loader warp w gathers the contiguous 4 KiB
// slice [4096 w, 4096 w + 4096) of the chunk with 16-byte streaming loads,
// XORs old and new, counts changes, and sets one bitmap bit per non-zero mask
// byte.  The next chunk's ticket, descriptor and pieces are staged one
// iteration ahead, so the data loads of a chunk issue at once.  Encoder warp
// b owns buffer b: it compacts the bitmap into a sorted list of non-zero byte
// positions ("events"), parses the chunk from the events 32 at a time (one per
// lane, connected by warp scans), waits for its place in the stream and writes
// the frame, while the loaders fill the other buffer.  Named barriers hand the
// buffers back and forth.
//
// LZ4 parse.  The masks are long zero runs around sparse non-zero bytes, so
// every zero run of at least 4 bytes becomes one match and everything else
// stays literal.  A run is copied from the longest earlier zero run when that
// one is long enough (non-overlapping copy), else it keeps its first zero as a
// literal and copies from it with offset 1.  Every match therefore copies zero
// bytes only (frame flag ZSRC), and the block obeys the format's end rules
// (last 5 bytes literals, no match start in the last 12 bytes).
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "dcr_internal.h"

namespace dcr {
namespace {

constexpr int kLoaders = 16;                      // loader warps
constexpr int kEncoders = 2;                      // encoder warps = chunk buffers
constexpr int kThreads = 32 * (kLoaders + kEncoders);
constexpr int kLoaderThreads = 32 * kLoaders;
constexpr int kNVec = kChunk / 16;                // 16-byte vectors per chunk
constexpr int kVecPerWarp = kNVec / kLoaders;     // 256: a 4 KiB slice
constexpr int kVPL = kVecPerWarp / 32;            // 8 vectors per lane
constexpr int kWords = kChunk / 32;               // bitmap words per chunk
constexpr int kSteps = kWords / 32;               // 64 warp steps over the bitmap
constexpr int kEvCap = 6144;                      // events listed per batch
constexpr int kSegCache = 64;                     // sender pieces staged in smem
constexpr uint32_t kEnd = 0xFFFFFFFFu;
constexpr uint32_t kSpinLimit = 1u << 22;         // bounded look-back wait

// named barriers (0 is left to __syncthreads, unused here)
constexpr int kBarLoaders = 1;
constexpr int kBarEmpty = 2;                   // + buffer
constexpr int kBarFull = 2 + kEncoders;        // + buffer

struct EncArgs {
    const ChunkDesc* chunks;
    const Seg* src;
    const uint8_t* olds[DCR_MAX_TP];
    const uint8_t* news[DCR_MAX_TP];
    uint32_t chunk_begin, chunk_count;
    uint32_t mode;
    uint8_t* payload;
    uint64_t cap;
    EncScratch* sc;
    unsigned long long* counts;
    uint64_t* lb;
    uint32_t* fsize;
};

// chunk metadata staged in shared memory
struct __align__(16) Meta {
    ChunkDesc cd;
    uint32_t k;                        // window-relative chunk, or kEnd
    uint32_t pad[3];
    Seg segs[kSegCache];               // first pieces (all of them if src_count <= kSegCache)
};

struct __align__(16) Buf {
    uint4 data[kNVec];                 // mask (XOR chunks) or new bytes (overwrite chunks)
    uint32_t bits[kWords];             // bit i set iff mask byte i != 0
    uint16_t ev[kEvCap + 16];          // event list (sorted non-zero byte positions)
    uint32_t chg[kLoaders];            // changed stored values per slice
    Meta meta;
};

struct __align__(16) Smem {
    Buf buf[kEncoders];
    Meta next;                         // the loaders' next chunk, staged ahead
};

// ---------------------------------------------------------------- helpers --
__device__ __forceinline__ uint4 ld_stream(const void* p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void st_release(uint64_t* p, uint64_t v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ uint64_t ld_acquire(const uint64_t* p)
{
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void bar_sync(int id, int n)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void bar_arrive(int id, int n)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// 4-bit mask of the non-zero bytes of w (bit i <-> byte i)
__device__ __forceinline__ uint32_t nz4(uint32_t w)
{
    uint32_t t = __vcmpne4(w, 0u) & 0x01010101u;
    return (t * 0x01020408u) >> 24;
}

__device__ __forceinline__ uint32_t nz16(uint4 v)
{
    return nz4(v.x) | (nz4(v.y) << 4) | (nz4(v.z) << 8) | (nz4(v.w) << 12);
}

// changed stored values in a 16-byte mask vector with non-zero-byte mask m
// (bf16: 16-bit words; e4m3: bytes; e2m1: nibbles)
__device__ __forceinline__ uint32_t changed_in(uint32_t m, uint4 v, uint32_t bits)
{
    if (bits == 16) return __popc((m | (m >> 1)) & 0x5555u);
    if (bits == 8) return __popc(m);
    uint32_t c = 0;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t t = w[i] | (w[i] >> 1);
        t |= t >> 2;
        c += __popc(t & 0x11111111u);
    }
    return c;
}

// overwrite units of a bitmap word: bit i set iff the unit starting at byte i
// (ub = 2: even i only) has a non-zero mask byte
__device__ __forceinline__ uint32_t unit_bits(uint32_t b, uint32_t ub)
{
    return ub == 2 ? (b | (b >> 1)) & 0x55555555u : b;
}

// piece of the chunk holding canonical byte x: last piece with off <= x
__device__ __forceinline__ int find_seg(const Seg* s, int n, uint32_t x)
{
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (s[mid].off <= x) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ uint32_t ext_len(uint32_t n)   // extra length bytes
{
    return n < 15 ? 0u : 1u + (n - 15) / 255;
}

__device__ __forceinline__ uint32_t seq_bytes(uint32_t ll, uint32_t ml)
{
    return 1 + ext_len(ll) + ll + 2 + ext_len(ml - 4);
}

// ---- warp scans -------------------------------------------------------------
__device__ __forceinline__ uint32_t warp_incl_sum(uint32_t v, int lane)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v += o;
    }
    return v;
}

__device__ __forceinline__ unsigned long long warp_incl_max64(unsigned long long v, int lane)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        unsigned long long o = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d && o > v) v = o;
    }
    return v;
}

__device__ __forceinline__ int warp_incl_max(int v, int lane)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, v, d);
        if (lane >= d) v = max(v, o);
    }
    return v;
}

// ---- events -------------------------------------------------------------------
// Appends the positions of the set bits of bitmap steps [t, ...) to B.ev,
// in order, until a further step might not fit.  Returns the step reached.
__device__ __forceinline__ int list_events(Buf& B, int t, int lane, int* n_out)
{
    int n = 0;
    for (; t < kSteps; ++t) {
        const uint32_t w = B.bits[32 * t + lane];
        const uint32_t c = __popc(w);
        const uint32_t incl = warp_incl_sum(c, lane);
        const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
        if (n + int(tot) > kEvCap) break;
        uint32_t at = uint32_t(n) + incl - c, b = w;
        while (b) {
            const int i = __ffs(b) - 1;
            b &= b - 1;
            B.ev[at++] = uint16_t((32 * t + lane) * 32 + i);
        }
        n += int(tot);
    }
    __syncwarp();
    *n_out = n;
    return t;
}

// Carried parse state between groups of 32 events.
struct Parse {
    int prev;                  // last non-zero byte so far (-1: before the chunk)
    unsigned long long best;   // longest zero run of earlier groups: len << 32 | start
    int lit;                   // end of the last match (start of pending literals)
    uint32_t out;              // block bytes so far
};

// Zero-run parse of n listed events (plus the virtual event at raw when
// final), 32 at a time, one per lane.  A run copies from the longest zero run
// of the earlier groups, so every lane decides with carried state only; the
// literal start of a match is the end of the nearest earlier match, found with
// one ballot.  With body != nullptr the sequences are also written.
__device__ __forceinline__ void parse_events(const Buf& B, int n, bool final, int raw, Parse& P,
                                             uint8_t* body, uint32_t body_len, int lane, bool* bad)
{
    const uint8_t* bytes = reinterpret_cast<const uint8_t*>(B.data);
    const int total = n + (final ? 1 : 0);
    const uint32_t lt = (1u << lane) - 1u;
    for (int g = 0; g < total; g += 32) {
        const int i = g + lane;
        const bool active = i < total;
        const bool last = final && i == total - 1;
        const int p = !active ? raw : (last ? raw : int(B.ev[i]));
        int pp = __shfl_up_sync(0xffffffffu, p, 1);
        if (lane == 0) pp = P.prev;
        const int gs = pp + 1;
        const int L = p - gs;
        const int me = p < raw - 5 ? p : raw - 5;
        const uint32_t bl = uint32_t(P.best >> 32);
        const int bs = int(uint32_t(P.best));
        int ms = -1, off = 0;
        if (active && L > 0) {
            if (me - gs >= 4 && gs <= raw - 12 && bl >= uint32_t(me - gs)) {
                ms = gs;
                off = gs - bs;
            } else if (me - gs - 1 >= 4 && gs + 1 <= raw - 12) {
                ms = gs + 1;
                off = 1;
            }
        }
        const bool has = ms >= 0;
        const uint32_t M = __ballot_sync(0xffffffffu, has);
        const uint32_t below = M & lt;
        const int src = below ? 31 - __clz(below) : lane;
        int lit = __shfl_sync(0xffffffffu, me, src);
        if (!below) lit = P.lit;
        uint32_t sz = has ? seq_bytes(uint32_t(ms - lit), uint32_t(me - ms)) : 0u;
        const int flit = has ? me : lit;    // literals after this event's match
        if (last) sz += 1 + ext_len(uint32_t(raw - flit)) + uint32_t(raw - flit);
        uint32_t gsum;
        if (body) {
            const uint32_t incl = warp_incl_sum(sz, lane);
            gsum = __shfl_sync(0xffffffffu, incl, 31);
            if (has || last) {
                const uint32_t o0 = P.out + incl - sz;
                uint32_t o = o0;
                const uint32_t end = o0 + sz < body_len ? o0 + sz : body_len;
                auto put = [&](uint32_t v) {
                    if (o < end) body[o] = uint8_t(v);
                    ++o;
                };
                auto put_len = [&](uint32_t v) {
                    v -= 15;
                    for (; v >= 255; v -= 255) put(255);
                    put(v);
                };
                if (has) {
                    const uint32_t ll = uint32_t(ms - lit), mc = uint32_t(me - ms - 4);
                    put(((ll >= 15 ? 15u : ll) << 4) | (mc >= 15 ? 15u : mc));
                    if (ll >= 15) put_len(ll);
                    for (uint32_t q = 0; q < ll; ++q) put(bytes[lit + int(q)]);
                    put(uint32_t(off) & 0xFFu);
                    put(uint32_t(off) >> 8);
                    if (mc >= 15) put_len(mc);
                }
                if (last) {
                    const uint32_t ll = uint32_t(raw - flit);
                    put((ll >= 15 ? 15u : ll) << 4);
                    if (ll >= 15) put_len(ll);
                    for (uint32_t q = 0; q < ll; ++q) put(bytes[flit + int(q)]);
                }
                if (o != o0 + sz || o > body_len) *bad = true;
            }
        } else {
            gsum = __reduce_add_sync(0xffffffffu, sz);
        }
        // carry to the next group
        const int lastlane = (total - g < 32 ? total - g : 32) - 1;
        P.prev = __shfl_sync(0xffffffffu, p, lastlane);
        const uint32_t clen = active && L > 0 ? uint32_t(L) : 0u;
        const uint32_t mlen = __reduce_max_sync(0xffffffffu, clen);
        const uint32_t mst = __reduce_max_sync(0xffffffffu, clen == mlen && mlen ? uint32_t(gs) : 0u);
        const unsigned long long gbest = ((unsigned long long)mlen << 32) | mst;
        if (gbest > P.best) P.best = gbest;
        if (M) P.lit = __shfl_sync(0xffffffffu, me, 31 - __clz(M));
        P.out += gsum;
    }
}

// LZ4 block size (pass 1) or block bytes (pass 2) of the chunk in B.
// Events that fit are listed once; larger event sets are listed in batches.
__device__ uint32_t lz4_block(Buf& B, int raw, uint8_t* body, uint32_t body_len, bool reuse, int n_reuse,
                              int lane, bool* bad, int* n_listed, bool* complete)
{
    Parse P{-1, 0ull, 0, 0u};
    if (reuse) {
        parse_events(B, n_reuse, true, raw, P, body, body_len, lane, bad);
        return P.out;
    }
    int t = 0, n = 0;
    bool first = true;
    while (true) {
        t = list_events(B, t, lane, &n);
        const bool fin = t >= kSteps;
        if (first) {
            *n_listed = n;
            *complete = fin;
            first = false;
        }
        parse_events(B, n, fin, raw, P, body, body_len, lane, bad);
        if (fin) break;
    }
    return P.out;
}

// ---------------------------------------------------------------- loaders --
// Gather, XOR, count and map one chunk's 4 KiB slice (loader warp w).
// between() runs after the slice's loads are issued, before they are used.
template <class Between>
__device__ __forceinline__ void load_slice(const EncArgs& A, Buf& B, const Meta& M, bool overwrite,
                                           int w, int lane, Between between)
{
    const ChunkDesc& cd = M.cd;
    const int raw = int(cd.raw_len);
    const int nseg = int(cd.src_count);
    const Seg* segs = nseg <= kSegCache ? M.segs : A.src + cd.src_begin;
    uint8_t* bytes = reinterpret_cast<uint8_t*>(B.data);
    uint32_t changed = 0;
    const int v0 = w * kVecPerWarp;

    // bitmap word of the vector pair (v, v + 1) held by lanes (even, odd)
    auto map_vec = [&](int v, uint32_t z) {
        const uint32_t hi = __shfl_down_sync(0xffffffffu, z, 1);
        if ((lane & 1) == 0) B.bits[v >> 1] = z | (hi << 16);
    };

    if (cd.flags & kSrcVec) {
        const int nvec = raw >> 4;
        uint4 o[kVPL], n[kVPL];
        int cur = 0;
#pragma unroll
        for (int j = 0; j < kVPL; ++j) {
            const int v = v0 + j * 32 + lane;
            o[j] = n[j] = make_uint4(0, 0, 0, 0);
            if (v < nvec) {
                const uint32_t x = uint32_t(v) << 4;
                if (nseg > 1) {
                    if (j == 0) cur = find_seg(segs, nseg, x);
                    while (cur + 1 < nseg && segs[cur + 1].off <= x) ++cur;
                }
                const Seg sg = segs[cur];
                const uint32_t r = uint32_t(sg.addr >> kShardShift);
                const uint64_t a = (sg.addr & kAddrMask) + (x - sg.off);
                o[j] = ld_stream(A.olds[r] + a);
                n[j] = ld_stream(A.news[r] + a);
            }
        }
        between();
#pragma unroll
        for (int j = 0; j < kVPL; ++j) {
            const int v = v0 + j * 32 + lane;
            uint4 m = make_uint4(o[j].x ^ n[j].x, o[j].y ^ n[j].y, o[j].z ^ n[j].z, o[j].w ^ n[j].w);
            uint32_t z = nz16(m);
            changed += changed_in(z, m, cd.bits);
            B.data[v] = overwrite ? n[j] : m;
            map_vec(v, z);
        }
    } else {
        // unaligned pieces: byte-wise gather (layouts with odd row sizes).
        // The mask is staged first; overwrite chunks then restage new bytes.
        between();
        for (int pass = 0; pass < (overwrite ? 2 : 1); ++pass) {
            for (int i = lane; i < 16 * kVecPerWarp; i += 32) {
                const int x = 16 * v0 + i;
                uint8_t ob = 0, nb = 0;
                if (x < raw) {
                    const Seg sg = segs[find_seg(segs, nseg, uint32_t(x))];
                    const uint32_t r = uint32_t(sg.addr >> kShardShift);
                    const uint64_t a = (sg.addr & kAddrMask) + (uint32_t(x) - sg.off);
                    ob = A.olds[r][a];
                    nb = A.news[r][a];
                }
                bytes[x] = pass == 1 ? nb : uint8_t(ob ^ nb);
            }
            __syncwarp();
            if (pass == 0) {
                for (int j = 0; j < kVPL; ++j) {
                    const int v = v0 + j * 32 + lane;
                    const uint4 m = B.data[v];
                    const uint32_t z = nz16(m);
                    changed += changed_in(z, m, cd.bits);
                    map_vec(v, z);
                }
                __syncwarp();
            }
        }
    }
    changed = __reduce_add_sync(0xffffffffu, changed);
    if (lane == 0) B.chg[w] = changed;
}

// Loader warp 0: stage the next chunk's descriptor and pieces.  `ticket`
// (lane 0) holds the chunk taken one call earlier; a new one is taken here.
__device__ __forceinline__ void stage_next(const EncArgs& A, Meta& M, int lane, uint32_t& ticket)
{
    uint32_t k = 0;
    if (lane == 0) {
        k = ticket;
        if (k >= A.chunk_count || *(volatile int32_t*)&A.sc->err) k = kEnd;
        if (k != kEnd) ticket = atomicAdd(&A.sc->ticket, 1u);
    }
    k = __shfl_sync(0xffffffffu, k, 0);
    if (lane == 0) M.k = k;
    if (k == kEnd) return;
    const ChunkDesc cd = A.chunks[A.chunk_begin + k];
    if (lane == 0) M.cd = cd;
    const uint32_t ns = cd.src_count < uint32_t(kSegCache) ? cd.src_count : uint32_t(kSegCache);
    for (uint32_t i = lane; i < ns; i += 32) M.segs[i] = A.src[cd.src_begin + i];
}

// ---------------------------------------------------------------- encoder --
// Parse, place and write the frame of the chunk held in buffer B.
__device__ __forceinline__ void encode_chunk(const EncArgs& A, Buf& B, int lane)
{
    const ChunkDesc cd = B.meta.cd;
    const uint32_t k = B.meta.k;
    const int raw = int(cd.raw_len);
    const bool overwrite = (cd.flags & kResidualFlag) || A.mode == DCR_MODE_OVERWRITE_ONLY;
    const uint8_t* bytes = reinterpret_cast<const uint8_t*>(B.data);

    uint32_t chg = lane < kLoaders ? B.chg[lane] : 0u;
    chg = __reduce_add_sync(0xffffffffu, chg);
    if (lane == 0 && chg) {
        atomicAdd(&A.counts[cd.tensor], (unsigned long long)chg);
        atomicAdd(reinterpret_cast<unsigned long long*>(&A.sc->changed), (unsigned long long)chg);
    }

    uint32_t kind = 0, body_len = 0, n_units = 0;
    int n_listed = 0;
    bool complete = false, bad = false;
    const uint32_t ub = cd.bits == 16 ? 2u : 1u;
    if (chg && !overwrite) {
        const uint32_t total = lz4_block(B, raw, nullptr, 0, false, 0, lane, &bad, &n_listed, &complete);
        if (total < uint32_t(raw)) {
            kind = kXorLz4;
            body_len = total;
        } else {
            kind = kXorRaw;
            body_len = uint32_t(raw);
        }
    } else if (chg) {
        // overwrite records: one per changed unit (2 bytes for bf16, else 1)
        uint32_t units = 0;
        for (int t = 0; t < kSteps; ++t) units += __popc(unit_bits(B.bits[32 * t + lane], ub));
        n_units = __reduce_add_sync(0xffffffffu, units);
        const uint32_t pad = (4 - (2 * n_units) % 4) % 4;
        const uint32_t rec = 4 + 2 * n_units + pad + n_units * ub;
        if (rec < uint32_t(raw)) {
            kind = kOverwrite;
            body_len = rec;
        } else {
            kind = kOverwriteDense;
            body_len = uint32_t(raw);
        }
    }
    const uint32_t fsz = chg ? (kFrameHdr + body_len + 15) / 16 * 16 : 0u;

    // ---- decoupled look-back for the frame's place in the stream: the warp
    // reads 32 predecessors per round trip, newest first, and sums them up to
    // the nearest one that already holds an inclusive prefix
    uint64_t excl = 0;
    int ok = 1;
    const uint64_t agg = fsz ? ((1ull << kLbFrameShift) | fsz) : 0ull;
    if (lane == 0) {
        A.fsize[k] = fsz;
        st_release(&A.lb[k], (k == 0 ? kLbInc : kLbAgg) | agg);
    }
    if (k > 0) {
        for (int64_t j = int64_t(k) - 1;; j -= 32) {
            const int64_t idx = j - lane;
            uint64_t v = 0;
            uint32_t spins = 0;
            for (;;) {
                v = idx >= 0 ? ld_acquire(&A.lb[idx]) : kLbInc;   // before chunk 0: prefix 0
                const uint32_t inc = __ballot_sync(0xffffffffu, (v >> 62) == 2);
                const uint32_t upto = inc ? (2u << (__ffs(inc) - 1)) - 1u : 0xffffffffu;
                const uint32_t missing = __ballot_sync(0xffffffffu, (v >> 62) == 0) & upto;
                if (!missing) break;
                const bool quit = ++spins > kSpinLimit || *(volatile int32_t*)&A.sc->err != 0;
                if (__any_sync(0xffffffffu, quit)) {   // warp-uniform exit
                    ok = 0;
                    break;
                }
                __nanosleep(64);
            }
            if (!ok) break;
            const uint32_t inc = __ballot_sync(0xffffffffu, (v >> 62) == 2);
            const uint32_t upto = inc ? (2u << (__ffs(inc) - 1)) - 1u : 0xffffffffu;
            uint64_t part = ((upto >> lane) & 1u) ? (v & kLbValMask) : 0ull;
#pragma unroll
            for (int d = 16; d > 0; d >>= 1) part += __shfl_xor_sync(0xffffffffu, part, d);
            excl += part;
            if (inc) break;
        }
        if (lane == 0) {
            if (ok) st_release(&A.lb[k], kLbInc | (excl + agg));
            else atomicCAS(reinterpret_cast<int*>(&A.sc->err), 0, DCR_ERR_TIMEOUT);
        }
    }
    if (!ok) return;

    // ---- write the frame
    const uint64_t foff = kStreamHdr + (excl & kLbByteMask);
    if (!fsz || foff + fsz > A.cap) return;
    uint8_t* f = A.payload + foff;
    uint8_t* body = f + kFrameHdr;
    if (lane == 0) {
        const uint32_t h1 = kind | (cd.bits << 8) | ((kind == kXorLz4 ? kFrameZsrc : 0u) << 16);
        reinterpret_cast<uint4*>(f)[0] = make_uint4(kFrameMagic, h1, A.chunk_begin + k, uint32_t(raw));
        reinterpret_cast<uint4*>(f)[1] = make_uint4(body_len, chg, 0u, 0u);
    }
    for (uint32_t i = kFrameHdr + body_len + lane; i < fsz; i += 32) f[i] = 0;
    if (kind == kXorLz4) {
        int nl;
        bool cp;
        const uint32_t got = lz4_block(B, raw, body, body_len, complete, n_listed, lane, &bad, &nl, &cp);
        if (__any_sync(0xffffffffu, bad) || got != body_len)   // sizing and emission disagree
            if (lane == 0) atomicCAS(reinterpret_cast<int*>(&A.sc->err), 0, DCR_ERR_CORRUPT);
    } else if (kind == kXorRaw || kind == kOverwriteDense) {
        const int nfull = raw >> 4;
        for (int v = lane; v < nfull; v += 32) reinterpret_cast<uint4*>(body)[v] = B.data[v];
        for (int x = (nfull << 4) + lane; x < raw; x += 32) body[x] = bytes[x];
    } else {
        const uint32_t pad = (4 - (2 * n_units) % 4) % 4;
        if (lane == 0) {
            *reinterpret_cast<uint32_t*>(body) = n_units;
            for (uint32_t i = 0; i < pad; ++i) body[4 + 2 * n_units + i] = 0;
        }
        uint8_t* offs = body + 4;
        uint8_t* vals = body + 4 + 2 * n_units + pad;
        uint32_t base = 0;
        for (int t = 0; t < kSteps; ++t) {
            const int wi = 32 * t + lane;
            uint32_t b = unit_bits(B.bits[wi], ub);
            const uint32_t c = __popc(b);
            const uint32_t incl = warp_incl_sum(c, lane);
            uint32_t u_i = base + incl - c;
            while (b) {
                const uint32_t x = uint32_t(wi * 32 + __ffs(b) - 1);
                b &= b - 1;
                const uint32_t u = x / ub;
                if (u_i < n_units) {
                    offs[2 * u_i] = uint8_t(u);
                    offs[2 * u_i + 1] = uint8_t(u >> 8);
                    for (uint32_t e = 0; e < ub; ++e) vals[u_i * ub + e] = bytes[x + e];
                }
                ++u_i;
            }
            base += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
}

// ================================================================ kernel ==
__global__ void __launch_bounds__(kThreads, 1) encode_kernel(EncArgs A)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem& S = *reinterpret_cast<Smem*>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp >= kLoaders) {
        // encoder warp: owns buffer b
        const int b = warp - kLoaders;
        Buf& B = S.buf[b];
        __threadfence_block();
        bar_arrive(kBarEmpty + b, kLoaderThreads + 32);
        for (;;) {
            bar_sync(kBarFull + b, kLoaderThreads + 32);
            if (B.meta.k == kEnd) break;
            encode_chunk(A, B, lane);
            __syncwarp();
            __threadfence_block();
            bar_arrive(kBarEmpty + b, kLoaderThreads + 32);
        }
        return;
    }

    // loader warps.  Warp 0 stages each chunk's ticket, descriptor and
    // pieces one iteration ahead, so they are in shared memory when the
    // chunk's loads issue.
    uint32_t ticket = 0;
    if (threadIdx.x == 0) ticket = atomicAdd(&A.sc->ticket, 1u);
    if (warp == 0) stage_next(A, S.next, lane, ticket);
    bar_sync(kBarLoaders, kLoaderThreads);
    for (int b = 0;; b = b + 1 == kEncoders ? 0 : b + 1) {
        Buf& B = S.buf[b];
        bar_sync(kBarEmpty + b, kLoaderThreads + 32);
        if (warp == 0) {
            if (lane == 0) {
                B.meta.k = S.next.k;
                B.meta.cd = S.next.cd;
            }
            const uint32_t ns = S.next.k == kEnd ? 0u
                : (S.next.cd.src_count < uint32_t(kSegCache) ? S.next.cd.src_count : uint32_t(kSegCache));
            for (uint32_t i = lane; i < ns; i += 32) B.meta.segs[i] = S.next.segs[i];
        }
        bar_sync(kBarLoaders, kLoaderThreads);
        const uint32_t k = B.meta.k;
        if (k == kEnd) {
            // no chunk left: release every encoder warp, each once it is idle
            __threadfence_block();
            bar_arrive(kBarFull + b, kLoaderThreads + 32);
            for (int d = 1; d < kEncoders; ++d) {
                const int o = (b + d) % kEncoders;
                bar_sync(kBarEmpty + o, kLoaderThreads + 32);
                if (threadIdx.x == 0) S.buf[o].meta.k = kEnd;
                __threadfence_block();
                bar_arrive(kBarFull + o, kLoaderThreads + 32);
            }
            break;
        }
        const bool overwrite = (B.meta.cd.flags & kResidualFlag) || A.mode == DCR_MODE_OVERWRITE_ONLY;
        // warp 0 stages the next chunk while this chunk's loads are in flight
        load_slice(A, B, B.meta, overwrite, warp, lane, [&] {
            if (warp == 0) stage_next(A, S.next, lane, ticket);
        });
        __threadfence_block();
        bar_arrive(kBarFull + b, kLoaderThreads + 32);
    }
}

// Frame index and stream header, once every chunk's prefix is known.
__global__ void finalize_kernel(EncArgs A, uint64_t plan_hash, uint64_t base_v, uint64_t target_v,
                                uint32_t window)
{
    if (*(volatile int32_t*)&A.sc->err) return;
    const uint64_t last = ld_acquire(&A.lb[A.chunk_count - 1]) & kLbValMask;
    const uint64_t fbytes = last & kLbByteMask, nframes = last >> kLbFrameShift;
    const uint64_t total = kStreamHdr + fbytes + 8 * nframes;
    const bool fits = total <= A.cap;
    uint64_t* index = reinterpret_cast<uint64_t*>(A.payload + kStreamHdr + fbytes);
    for (uint32_t k = blockIdx.x * blockDim.x + threadIdx.x; k < A.chunk_count;
         k += gridDim.x * blockDim.x) {
        uint32_t fs = A.fsize[k];
        if (!fs || !fits) continue;
        uint64_t inc = A.lb[k] & kLbValMask;
        index[(inc >> kLbFrameShift) - 1] = kStreamHdr + (inc & kLbByteMask) - fs;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        A.sc->total = total;
        A.sc->n_frames = nframes;
        if (fits) {
            uint32_t h[16];
            h[0] = kStreamMagic;
            h[1] = kFormat;
            h[2] = uint32_t(plan_hash);
            h[3] = uint32_t(plan_hash >> 32);
            h[4] = uint32_t(base_v);
            h[5] = uint32_t(base_v >> 32);
            h[6] = uint32_t(target_v);
            h[7] = uint32_t(target_v >> 32);
            h[8] = window;
            h[9] = A.mode == DCR_MODE_OVERWRITE_ONLY ? kStreamOverwriteOnly : 0u;
            h[10] = A.chunk_begin;
            h[11] = A.chunk_count;
            h[12] = uint32_t(nframes);
            h[13] = uint32_t(nframes >> 32);
            h[14] = uint32_t(total);
            h[15] = uint32_t(total >> 32);
            uint4* d = reinterpret_cast<uint4*>(A.payload);
            for (int i = 0; i < 4; ++i) d[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
        }
    }
}

}  // namespace

int encode_kernel_config(KernelConfig* kc)
{
    int dev;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&kc->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(encode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sizeof(Smem)));
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&kc->enc_blocks_per_sm, encode_kernel, kThreads,
                                                          sizeof(Smem));
    if (e != cudaSuccess) return cuda_error(e, "encode kernel configuration");
    if (kc->enc_blocks_per_sm < 1) return set_error(DCR_ERR_CUDA, "encode kernel does not fit on an SM");
    return DCR_OK;
}

int encode_launch(const dcr_plan* P, uint32_t mode, uint32_t window, const void* const* olds,
                  const void* const* news, uint64_t base_v, uint64_t target_v, void* payload,
                  size_t cap, cudaStream_t s)
{
    EncArgs A{};
    A.chunks = P->d_chunks;
    A.src = P->d_src;
    for (uint32_t r = 0; r < P->tp && r < DCR_MAX_TP; ++r) {
        A.olds[r] = static_cast<const uint8_t*>(olds[r]);
        A.news[r] = static_cast<const uint8_t*>(news[r]);
    }
    A.chunk_begin = uint32_t(P->win_start[window]);
    A.chunk_count = uint32_t(P->win_start[window + 1] - P->win_start[window]);
    A.mode = mode;
    A.payload = static_cast<uint8_t*>(payload);
    A.cap = payload ? cap : 0;
    A.sc = static_cast<EncScratch*>(P->d_enc);
    A.counts = reinterpret_cast<unsigned long long*>(static_cast<char*>(P->d_enc) + sizeof(EncScratch));
    A.lb = P->d_lb;
    A.fsize = P->d_fsize;
    size_t reset = reinterpret_cast<char*>(P->d_lb) - static_cast<char*>(P->d_enc) + A.chunk_count * 8ull;
    cudaError_t e = cudaMemsetAsync(P->d_enc, 0, reset, s);
    if (e != cudaSuccess) return cuda_error(e, "encode scratch reset");
    unsigned grid = unsigned(P->kc.num_sms * P->kc.enc_blocks_per_sm);
    if (grid > A.chunk_count) grid = A.chunk_count;
    if (P->profiling) cudaEventRecord(P->ev[0], s);
    encode_kernel<<<grid, kThreads, sizeof(Smem), s>>>(A);
    if (P->profiling) cudaEventRecord(P->ev[1], s);
    unsigned fgrid = (A.chunk_count + 255) / 256;
    if (fgrid > 1024) fgrid = 1024;
    finalize_kernel<<<fgrid, 256, 0, s>>>(A, P->hash, base_v, target_v, window);
    if (P->profiling) cudaEventRecord(P->ev[2], s);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_error(e, "encode launch");
    return DCR_OK;
}

}  // namespace dcr
