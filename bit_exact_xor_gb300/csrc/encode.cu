// Sender hot path: per window, one persistent kernel encodes every chunk
// into per-chunk slots, a scan places the frames and writes the stream
// header, a copy pass moves the slots into the stream, and two more passes
// write the frame bodies that outgrew their slots.
//
// Per 64 KiB canonical chunk the encoder gathers old and new through the
// plan's shard->canonical pieces, forms mask = old XOR new, counts changed
// stored values, encodes the chunk (LZ4 block, raw mask, overwrite records or
// dense overwrite) and writes the frame to a slot of its own; once every
// frame size is known a scan places the frames in chunk order and a copy pass
// moves them into the stream.
//
// Method: "GPU-accelerated weight teleportation", "Delta update algebra"
// (mask = old XOR new on raw bits) and "A strong baseline with the
// Blackwell-native DE" (LZ4 block format); NeMo-DCR paper summary, "Input and
// change detection" (bitwise compare per owner shard), "Direct Projection",
// "Residual Conversion" and "Hybrid encoding and compression" (XOR masks for
// affine changes, overwrites for residual ones).
//
// encode_kernel.  One warp per chunk, chunks taken in ticket order, 24 warps
// per SM.  The warp streams its chunk in 1 KiB steps: cp.async copies old
// and new into a three-stage landing buffer in shared memory, so two steps
// are in flight while one is processed.  (A second instantiation with
// twelve stages and 2-warp CTAs serves windows with fewer chunks than warp
// slots.)  It XORs and counts, and appends the positions and values of the
// non-zero mask bytes ("events") to a ring in shared memory.  Every 32 events it runs one parse group (one event per
// lane, connected by ballots and warp sums) that writes the LZ4 sequences
// straight into the chunk's frame slot in device scratch.  Overwrite chunks
// write their records there instead.  A chunk whose body or pending literals
// outgrow the slot or the ring is sized all the same (the parse carries on
// without writing) and is listed for the restream pass.  No warp waits for
// another: frame sizes go to a per-chunk array.
//
// scan_kernel / copy_kernel.  One CTA per tile of 8192 chunks scans the
// tile's frame sizes into offsets, taking the tile's start from the tiles
// before it (a decoupled look-back), and the last tile writes the stream
// header; then one warp per chunk copies its slot to its place in the
// stream with 16-byte stores and writes its index entry.
//
// restream_kernel.  One warp per chunk whose body outgrew its slot (masks
// above a few percent change): it runs the chunk's stream loop again, now
// that the frame's offset and size are known, and the parse writes the body
// straight into the stream.  Same loop, same groups, so the sizes agree by
// construction (checked).  What it cannot write (raw and dense frames, LZ4
// chunks whose pending literals outgrow the event ring) it lists for
// spill_kernel.
//
// spill_kernel.  One CTA per chunk listed by restream_kernel: 16 warps
// gather the mask into shared memory (64 KiB plus a bitmap of its non-zero
// bytes), then one warp re-runs the same parse over the bitmap's event list,
// reading literal bytes from the mask, and writes the frame at its place in
// the stream; raw and dense frames are copied by the whole CTA.  All three
// encoders call the same parse_group with groups of 32 consecutive events
// from the first one, so their sizes agree by construction (a disagreement
// is reported).
//
// Parse (LZ4 blocks, or Snappy blocks with the plan's Snappy codec: the
// CodecLz4 / CodecSnappy policies below give each sequence's bytes; the
// kernels are instantiated per codec).  The masks are long zero runs around
// sparse non-zero bytes, so
// every zero run of at least 4 bytes becomes one match and everything else
// stays literal.  A run is copied from the longest zero run of the earlier
// groups when that one is long enough (non-overlapping copy), else it keeps
// its first zero as a literal and copies from it with offset 1.  Every match
// therefore copies zero bytes only (frame flag ZSRC), and the block obeys the
// format's end rules (last 5 bytes literals, no match start in the last 12).
#include <cuda_runtime.h>

#include <climits>
#include <cstddef>
#include <cstdint>

#include "dcr_internal.h"

namespace dcr {
namespace {

constexpr uint32_t kFull = 0xffffffffu;
// encode_kernel
constexpr int kMWarps = 6;                        // warps per CTA, one chunk each; 4 CTAs per SM
constexpr int kMThreads = 32 * kMWarps;
constexpr int kRing = 512;                        // event ring entries per warp (power of two)
constexpr int kAppend = 256;                      // events appended to the ring at most at once
constexpr int kStep = 1024;                       // bytes per step: 32 contiguous bytes per lane
constexpr int kNS = 3;                            // landing stages: kNS - 1 steps in flight
constexpr int kNSDeep = 12;                       // ... in the deep variant for windows of few chunks
constexpr int kDeepWarps = 2;                     // warps per CTA of the deep variant
constexpr int kMSegCache = 64;                    // sender pieces cached per warp
constexpr uint32_t kSlotBody = kEncSlot - kFrameHdr;   // frame body bytes a slot holds
// spill_kernel
constexpr int kSWarps = 16;                       // each gathers one 4 KiB slice
constexpr int kSThreads = 32 * kSWarps;
constexpr int kNVec = kChunk / 16;                // 16-byte vectors per chunk
constexpr int kVecPerWarp = kNVec / kSWarps;      // 256
constexpr int kVPL = kVecPerWarp / 32;            // 8 vectors per lane
constexpr int kWords = kChunk / 32;               // bitmap words per chunk
constexpr int kSteps = kWords / 32;               // 64 warp steps over the bitmap
constexpr int kEvCap = 6144;                      // events listed per batch
constexpr int kSegCache = 64;

struct EncArgs {
    const ChunkDesc* chunks;
    const Seg* src;
    const uint8_t* olds[DCR_MAX_TP];
    const uint8_t* news[DCR_MAX_TP];
    uint32_t chunk_begin, chunk_count;
    uint32_t mode;
    uint8_t* payload;          // the stream (header written by scan_kernel when `header`), or null
    uint64_t cap;
    uint8_t* frames;           // where frame bytes go: frame at relative offset o -> frames + o
    uint64_t frame_base;       // index entry of that frame: frame_base + o
    uint64_t* index;           // the frames' index entries (null: at the end of `payload`)
    uint32_t header;
    uint8_t* ovf;              // per-warp overflow buffers (kOvfBytes each; null: none)
    uint8_t* heap;             // rests of bodies past their slots
    uint64_t heap_cap;
    uint64_t* heapoff;         // per chunk: where its rest sits in the heap
    const uint8_t* in;         // dcr_encode_retry: the XOR stream read
    uint64_t in_idx;           // ... its index offset
    uint64_t in_frames;        // ... and frame count
    EncScratch* sc;
    unsigned long long* counts;
    uint64_t* lb;              // frame offsets: frames before << 40 | bytes before
    uint32_t* fsize;           // frame size (| kSpilled), 0: no frame
    SpillRec* spill;
    uint32_t* deep;            // spill records left to spill_kernel
    uint8_t* slots;            // kEncSlot bytes per chunk
    uint32_t stall;            // test only: scan tile 0 never publishes its total
};

// encode_kernel: one warp's shared memory with NS landing stages
template <int NS>
struct __align__(16) WarpSmemT {
    uint4 land[NS][2][64];             // landing stages [stage][old, new][16-byte slot]: the
                                       // step's bytes 32 L + 16 h in slot land_slot(L, h)
    uint16_t pos[kRing];               // event ring: byte position in the chunk
    uint8_t val[kRing];                //             mask byte
    Seg segs[kMSegCache];              // the chunk's sender pieces
};
using WarpSmem = WarpSmemT<kNS>;
using WarpSmemDeep = WarpSmemT<kNSDeep>;
// overwrite chunks keep their record values in the ring's storage
constexpr int kValStage = int(sizeof(uint16_t) + sizeof(uint8_t)) * kRing;
static_assert(offsetof(WarpSmem, val) == offsetof(WarpSmem, pos) + sizeof(uint16_t) * kRing,
              "ring storage is contiguous");
static_assert(offsetof(WarpSmemDeep, val) == offsetof(WarpSmemDeep, pos) + sizeof(uint16_t) * kRing,
              "ring storage is contiguous");
static_assert(kAppend + 31 <= kRing, "a spilled chunk's unparsed events fit the ring");

// spill_kernel: one chunk in shared memory
struct __align__(16) Meta {
    ChunkDesc cd;
    uint32_t pad[4];
    Seg segs[kSegCache];               // first pieces (all of them if src_count <= kSegCache)
};

struct __align__(16) Buf {
    uint4 data[kNVec];                 // mask (XOR chunks) or new bytes (overwrite chunks)
    uint32_t bits[kWords];             // bit i set iff mask byte i != 0
    uint16_t ev[kEvCap + 32];          // event list (sorted non-zero byte positions)
    Meta meta;
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

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem)
{
    const uint32_t sa = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async16_sa(uint32_t saddr, const void* gmem)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint4 xor4(uint4 a, uint4 b)
{
    return make_uint4(a.x ^ b.x, a.y ^ b.y, a.z ^ b.z, a.w ^ b.w);
}

// byte i (0..15) of v, without dynamic register indexing
__device__ __forceinline__ uint32_t byte_of(uint4 v, uint32_t i)
{
    const uint32_t w = i < 8 ? (i < 4 ? v.x : v.y) : (i < 12 ? v.z : v.w);
    return (w >> (8 * (i & 3))) & 0xFFu;
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

// 32 mask bytes (a: bytes 0-15, b: bytes 16-31): bit i set iff byte i is
// non-zero.  Per word, bit 7 of each byte is set iff the byte is non-zero
// (the low 7 bits plus 0x7F carry into bit 7, or bit 7 was set); one
// multiply then gathers the eight flags of two words into one byte.
__device__ __forceinline__ uint32_t nz32(uint4 a, uint4 b)
{
    auto hb = [](uint32_t w) { return (((w & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | w) & 0x80808080u; };
    auto pair = [&](uint32_t lo, uint32_t hi) { return ((hb(hi) | (hb(lo) >> 4)) * 0x00204081u) >> 24; };
    return pair(a.x, a.y) | (pair(a.z, a.w) << 8) | (pair(b.x, b.y) << 16) | (pair(b.z, b.w) << 24);
}

// byte i (0..31) of the 32 bytes (a, b)
__device__ __forceinline__ uint32_t byte_of32(uint4 a, uint4 b, uint32_t i)
{
    const uint4 v = (i & 16) ? b : a;
    return byte_of(v, i & 15);
}

// non-zero 4-bit nibbles of a word
__device__ __forceinline__ uint32_t nibbles_nz(uint32_t w)
{
    uint32_t t = w | (w >> 1);
    t |= t >> 2;
    return __popc(t & 0x11111111u);
}

// overwrite units of a non-zero-byte mask: bit i set iff the unit starting at
// byte i (ub = 2: even i only) has a non-zero mask byte
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

// Block codecs of the XOR masks.  Both encode the parse's sequences (a
// literal run, then a copy of zero bytes); only the byte layout differs.
//
// LZ4 block: per sequence a token (literal length << 4 | match length - 4,
// 15 = more length bytes of 255 follow), literals, a 2-byte offset, match
// length bytes; the last sequence is literals only.
struct CodecLz4 {
    static constexpr uint32_t kKind = kXorLz4;
    static constexpr bool kNearCopy = false;   // see CodecSnappy
    __device__ static uint32_t preamble(uint32_t) { return 0u; }
    __device__ static uint32_t seq(uint32_t ll, uint32_t ml, uint32_t) { return seq_bytes(ll, ml); }
    __device__ static uint32_t tail(uint32_t ll) { return 1 + ext_len(ll) + ll; }
    template <class Put>
    __device__ static void put_len(Put& put, uint32_t v)
    {
        v -= 15;
        for (; v >= 255; v -= 255) put(255);
        put(v);
    }
    // the sequence's bytes; lits(put) writes its literal bytes
    template <class Put, class Lits>
    __device__ static void emit_seq(Put& put, uint32_t ll, Lits&& lits, uint32_t off, uint32_t ml)
    {
        const uint32_t mc = ml - 4;
        put(((ll >= 15 ? 15u : ll) << 4) | (mc >= 15 ? 15u : mc));
        if (ll >= 15) put_len(put, ll);
        lits(put);
        put(off & 0xFFu);
        put(off >> 8);
        if (mc >= 15) put_len(put, mc);
    }
    template <class Put, class Lits>
    __device__ static void emit_tail(Put& put, uint32_t ll, Lits&& lits)
    {
        put((ll >= 15 ? 15u : ll) << 4);
        if (ll >= 15) put_len(put, ll);
        lits(put);
    }
    template <class Put>
    __device__ static void emit_preamble(Put&, uint32_t) {}
};

// Snappy block ("A strong baseline with the Blackwell-native DE", footnote
// 4): the chunk length as a base-128 varint, then literal elements (tag
// (length - 1) << 2 below 60, else 60..63 and 1..4 length bytes) and copy
// elements of at most 64 bytes (tag 1: length 4..11 and an 11-bit offset in
// 2 bytes; tag 2: length 1..64 and a 2-byte offset).  A match becomes copies
// of 64 while at least 68 bytes remain, one of 60 if more than 64 remain,
// then the rest (4 or more).
struct CodecSnappy {
    static constexpr uint32_t kKind = kXorSnappy;
    // a copy of 4..11 bytes at an offset below 2048 takes 2 bytes instead of
    // 3, so a run may also copy from the zero gap just before the previous
    // event (all bytes between two events are zero), usually close by
    static constexpr bool kNearCopy = true;
    __device__ static uint32_t preamble(uint32_t raw) { return raw < 128 ? 1u : raw < 16384 ? 2u : 3u; }
    __device__ static uint32_t lit_bytes(uint32_t ll)
    {
        return ll == 0 ? 0u : 1u + (ll <= 60 ? 0u : ll <= 256 ? 1u : ll <= 65536 ? 2u : 3u) + ll;
    }
    __device__ static uint32_t copy_bytes(uint32_t ml, uint32_t off)
    {
        const uint32_t k = ml >= 68 ? (ml - 68) / 64 + 1 : 0u;
        uint32_t r = ml - 64 * k, c = 3 * k;
        if (r > 64) {
            c += 3;
            r -= 60;
        }
        return c + (r <= 11 && off < 2048 ? 2u : 3u);
    }
    __device__ static uint32_t seq(uint32_t ll, uint32_t ml, uint32_t off) { return lit_bytes(ll) + copy_bytes(ml, off); }
    __device__ static uint32_t tail(uint32_t ll) { return lit_bytes(ll); }
    template <class Put, class Lits>
    __device__ static void emit_lits(Put& put, uint32_t ll, Lits&& lits)
    {
        if (ll) {
            const uint32_t v = ll - 1, nb = v < 60 ? 0u : v < 256 ? 1u : v < 65536 ? 2u : 3u;
            put((nb ? 59 + nb : v) << 2);
            for (uint32_t i = 0; i < nb; ++i) put((v >> (8 * i)) & 0xFFu);
        }
        lits(put);
    }
    template <class Put>
    __device__ static void emit_copy(Put& put, uint32_t len, uint32_t off)
    {
        if (len <= 11 && off < 2048) {
            put(1u | ((len - 4) << 2) | ((off >> 8) << 5));
            put(off & 0xFFu);
        } else {
            put(2u | ((len - 1) << 2));
            put(off & 0xFFu);
            put(off >> 8);
        }
    }
    template <class Put, class Lits>
    __device__ static void emit_seq(Put& put, uint32_t ll, Lits&& lits, uint32_t off, uint32_t ml)
    {
        emit_lits(put, ll, lits);
        for (; ml >= 68; ml -= 64) emit_copy(put, 64, off);
        if (ml > 64) {
            emit_copy(put, 60, off);
            ml -= 60;
        }
        emit_copy(put, ml, off);
    }
    template <class Put, class Lits>
    __device__ static void emit_tail(Put& put, uint32_t ll, Lits&& lits)
    {
        emit_lits(put, ll, lits);
    }
    template <class Put>
    __device__ static void emit_preamble(Put& put, uint32_t raw)
    {
        for (; raw >= 128; raw >>= 7) put((raw & 127u) | 128u);
        put(raw);
    }
};

__device__ __forceinline__ uint32_t warp_incl_sum(uint32_t v, int lane)
{
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_up_sync(kFull, v, d);
        if (lane >= d) v += o;
    }
    return v;
}

__device__ __forceinline__ void report(EncScratch* sc, int code)
{
    atomicCAS(reinterpret_cast<int*>(&sc->err), 0, code);
}

// ------------------------------------------------------------------ parse --
// Where a block's bytes go: Sink to one buffer; SplitSink bytes [0, split)
// to a, the rest to b (the slot, then a warp's overflow buffer).
struct Sink {
    uint8_t* a;
    __device__ __forceinline__ void put(uint32_t o, uint32_t v) const { a[o] = uint8_t(v); }
};
struct SplitSink {
    uint8_t* a;
    uint8_t* b;
    uint32_t split;
    __device__ __forceinline__ void put(uint32_t o, uint32_t v) const
    {
        if (o < split) a[o] = uint8_t(v);
        else b[o - split] = uint8_t(v);
    }
};

// Carried parse state between groups of 32 events.
struct Parse {
    int prev;                  // last non-zero byte so far (-1: before the chunk)
    unsigned long long best;   // longest zero run of earlier groups: len << 32 | start
    int lit;                   // end of the last match (start of pending literals)
    int lit_ev;                // first event at or after lit
    uint32_t out;              // block bytes so far
};

// Events of encode_kernel: the warp's ring of positions and mask bytes.
struct RingSrc {
    const uint16_t* pos;
    const uint8_t* val;
    __device__ __forceinline__ int at(int e) const { return pos[e & (kRing - 1)]; }
    // put the literal bytes [a, b), which hold events [e, e_end); false if
    // those events do not fall inside
    template <class Put>
    __device__ __forceinline__ bool lits(int a, int b, int e, int e_end, Put& put) const
    {
        for (int q = a; q < b; ++q) {
            uint32_t v = 0;
            if (e < e_end && int(pos[e & (kRing - 1)]) == q) {
                v = val[e & (kRing - 1)];
                ++e;
            }
            put(v);
        }
        return e == e_end;
    }
};

// Events of spill_kernel: the listed positions, literal bytes from the mask.
struct MaskSrc {
    const uint16_t* ev;
    const uint8_t* bytes;
    __device__ __forceinline__ int at(int e) const { return ev[e]; }
    template <class Put>
    __device__ __forceinline__ bool lits(int a, int b, int, int, Put& put) const
    {
        for (int q = a; q < b; ++q) put(bytes[q]);
        return true;
    }
};

// One parse group: events e0 .. e0 + cnt - 1, one per lane, plus the virtual
// event at raw when final (cnt + final <= 32).  A run copies from the longest
// zero run of the earlier groups, so every lane decides with carried state
// only; the literal start of a match is the end of the nearest earlier match,
// found with one ballot.  Sizes add up in P.out.  With emit, the sequences
// are written to out at [0, cap); *over is set when one does not fit and *bad
// when sizing and writing disagree.
// What a group's block bytes owe to the literal start carried in from the
// groups before it (parse_group's sizing pass can report it): only its first
// match's sequence and, in a final group without a match, the tail; the rest
// the group fixes by itself.
struct GroupSplit {
    uint32_t indep;      // bytes that do not depend on the carried literal start
    int ms0;             // the first match's start (-1: the group has none)
    uint32_t ml0, off0;  // ... its length and offset
    bool tail_dep;       // final group without a match: the tail's literals start there
};

template <class Codec, class Src, class Out = Sink>
__device__ __forceinline__ void parse_group(const Src& S, int e0, int cnt, bool final, int raw, Parse& P,
                                            const Out& out, uint32_t cap, bool emit, int lane, bool* over,
                                            bool* bad, GroupSplit* split = nullptr)
{
    const int total = cnt + (final ? 1 : 0);
    const uint32_t lt = (1u << lane) - 1u;
    const bool active = lane < total;
    const bool last = final && lane == total - 1;
    const int e = e0 + lane;
    const int p = (!active || last) ? raw : S.at(e);
    int pp = __shfl_up_sync(kFull, p, 1);
    if (lane == 0) pp = P.prev;
    const int gs = pp + 1;
    const int L = p - gs;
    if (!final && __all_sync(kFull, L == 0)) {
        // 32 back-to-back non-zero bytes: no zero run, no sequence, nothing
        // to carry but the last position
        P.prev = __shfl_sync(kFull, p, 31);
        return;
    }
    const int me = p < raw - 5 ? p : raw - 5;
    const uint32_t bl = uint32_t(P.best >> 32);
    const int bs = int(uint32_t(P.best));
    int ms = -1, off = 0;
    int pgs = 0, pL = 0;   // the previous lane's zero gap (Snappy)
    if constexpr (Codec::kNearCopy) {
        pgs = __shfl_up_sync(kFull, gs, 1);
        pL = __shfl_up_sync(kFull, L, 1);
    }
    if (Codec::kNearCopy && active && lane > 0 && L > 0 && me - gs >= 4 && gs <= raw - 12 && pL >= me - gs) {
        ms = gs;
        off = gs - pgs;
    } else if (active && L > 0) {
        if (me - gs >= 4 && gs <= raw - 12 && bl >= uint32_t(me - gs)) {
            ms = gs;
            off = gs - bs;
        } else if (me - gs - 1 >= 4 && gs + 1 <= raw - 12) {
            ms = gs + 1;
            off = 1;
        }
    }
    const bool has = ms >= 0;
    const uint32_t M = __ballot_sync(kFull, has);
    const uint32_t below = M & lt;
    const int src = below ? 31 - __clz(below) : lane;
    int lit = __shfl_sync(kFull, me, src);
    int lev = e0 + src;
    if (!below) {
        lit = P.lit;
        lev = P.lit_ev;
    }
    uint32_t sz = has ? Codec::seq(uint32_t(ms - lit), uint32_t(me - ms), uint32_t(off)) : 0u;
    const int flit = has ? me : lit;    // literals after this event's match
    if (last) sz += Codec::tail(uint32_t(raw - flit));
    uint32_t gsum;
    if (emit) {
        const uint32_t incl = warp_incl_sum(sz, lane);
        gsum = __shfl_sync(kFull, incl, 31);
        const uint32_t o0 = P.out + incl - sz;
        const bool fits = o0 + sz <= cap;
        if ((has || last) && !fits) *over = true;
        if ((has || last) && fits) {
            uint32_t o = o0;
            auto put = [&](uint32_t v) { out.put(o++, v); };
            bool ok = true;
            if (has)
                Codec::emit_seq(put, uint32_t(ms - lit), [&](decltype(put)& p) { ok &= S.lits(lit, ms, lev, e, p); },
                                uint32_t(off), uint32_t(me - ms));
            if (last)
                Codec::emit_tail(put, uint32_t(raw - flit),
                                 [&](decltype(put)& p) { ok &= S.lits(flit, raw, has ? e : lev, e, p); });
            if (!ok || o != o0 + sz) *bad = true;
        }
    } else {
        gsum = __reduce_add_sync(kFull, sz);
        if (split) {
            const bool dep = has && !below;            // the first match: literals from the carried start
            const bool tdep = last && !has && !below;  // no match in the group: nor the tail's
            const uint32_t tl = last ? Codec::tail(uint32_t(raw - flit)) : 0u;
            const uint32_t sq = sz - tl;
            split->indep = __reduce_add_sync(kFull, (dep ? 0u : sq) + (tdep ? 0u : tl));
            const int f = M ? __ffs(M) - 1 : 0;
            const int ms0 = __shfl_sync(kFull, ms, f);
            split->ms0 = M ? ms0 : -1;
            split->ml0 = uint32_t(__shfl_sync(kFull, me, f) - ms0);
            split->off0 = uint32_t(__shfl_sync(kFull, off, f));
            split->tail_dep = __any_sync(kFull, tdep);
        }
    }
    // carry to the next group
    P.prev = __shfl_sync(kFull, p, total - 1);
    const uint32_t clen = active && L > 0 ? uint32_t(L) : 0u;
    const uint32_t mlen = __reduce_max_sync(kFull, clen);
    const uint32_t mst = __reduce_max_sync(kFull, clen == mlen && mlen ? uint32_t(gs) : 0u);
    const unsigned long long gbest = ((unsigned long long)mlen << 32) | mst;
    if (gbest > P.best) P.best = gbest;
    if (M) {
        const int hi = 31 - __clz(M);
        P.lit = __shfl_sync(kFull, me, hi);
        P.lit_ev = e0 + hi;
    }
    P.out += gsum;
}

__device__ __forceinline__ void write_header(uint8_t* f, uint32_t kind, uint32_t bits, uint32_t chunk,
                                             uint32_t raw, uint32_t body_len, uint32_t chg)
{
    const uint32_t h1 = kind | (bits << 8) | ((kind == kXorLz4 || kind == kXorSnappy ? kFrameZsrc : 0u) << 16);
    reinterpret_cast<uint4*>(f)[0] = make_uint4(kFrameMagic, h1, chunk, raw);
    reinterpret_cast<uint4*>(f)[1] = make_uint4(body_len, chg, 0u, 0u);
}

// ---------------------------------------------------------- encode_kernel --
// Slot of the step's bytes [32 L + 16 h, + 16): the two halves of every
// fourth-lane group are swapped, so that lanes reading their own 32 bytes
// (one 16-byte load per half) hit distinct banks.
__device__ __forceinline__ int land_slot(int L, int h) { return 2 * L + (h ^ ((L >> 2) & 1)); }

// Byte-wise gather of one 16-byte vector at canonical byte x0 (chunks whose
// pieces are not all 16-byte aligned); bytes at or past raw read as zero.
__device__ __forceinline__ void gather_bytes(const EncArgs& A, const Seg* segs, int nseg, int& cur,
                                             uint32_t x0, int raw, uint4& o, uint4& n)
{
    uint32_t ow[4] = {0u, 0u, 0u, 0u}, nw[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int b = 0; b < 16; ++b) {
        const uint32_t x = x0 + uint32_t(b);
        if (x < uint32_t(raw)) {
            while (cur + 1 < nseg && segs[cur + 1].off <= x) ++cur;
            const Seg sg = segs[cur];
            const uint32_t r = uint32_t(sg.addr >> kShardShift);
            const uint64_t a = (sg.addr & kAddrMask) + (x - sg.off);
            ow[b >> 2] |= uint32_t(A.olds[r][a]) << (8 * (b & 3));
            nw[b >> 2] |= uint32_t(A.news[r][a]) << (8 * (b & 3));
        }
    }
    o = make_uint4(ow[0], ow[1], ow[2], ow[3]);
    n = make_uint4(nw[0], nw[1], nw[2], nw[3]);
}

// The stream loop of any chunk (overwrite records, 4-bit elements, pieces
// that are not 16-byte aligned); stream_fast below is the common case.
template <int NS, class Codec, class Out>
__device__ __forceinline__ void stream_chunk(const EncArgs& A, WarpSmemT<NS>& W, const ChunkDesc& cd, const Seg* segs,
                                             int lane, const Out& body, uint32_t cap, uint8_t* vals, int ncap,
                                             uint32_t& changed, Parse& P, int& tail, int& np, int& units,
                                             bool& spill, bool& bad)
{
    const int raw = int(cd.raw_len);
    const int nseg = int(cd.src_count);
    const bool overwrite = (cd.flags & kResidualFlag) || A.mode == DCR_MODE_OVERWRITE_ONLY;
    const bool vec = (cd.flags & kSrcVec) != 0;
    const uint32_t bits = cd.bits;
    const uint32_t ub = bits == 16 ? 2u : 1u;
    const int nsteps = (raw + kStep - 1) / kStep;
    const RingSrc R{W.pos, W.val};

    // step s of the chunk into landing stage s % NS (one commit group per
    // step); each copy instruction covers 512 contiguous bytes
    int cur = 0;
    auto issue = [&](int s) {
        if (s < nsteps) {
            const uint32_t x0 = uint32_t(s) * kStep;
            {
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    const uint32_t q = 512u * g + 16u * lane;   // byte of the step
                    const uint32_t x = x0 + q;
                    const int slot = land_slot(int(q >> 5), int(lane & 1));
                    uint4* lo = &W.land[s % NS][0][slot];
                    uint4* ln = &W.land[s % NS][1][slot];
                    if (x >= uint32_t(raw)) {
                        *lo = *ln = make_uint4(0u, 0u, 0u, 0u);
                    } else if (vec) {
                        while (cur + 1 < nseg && segs[cur + 1].off <= x) ++cur;
                        const Seg sg = segs[cur];
                        const uint32_t r = uint32_t(sg.addr >> kShardShift);
                        const uint64_t a = (sg.addr & kAddrMask) + (x - sg.off);
                        cp_async16(lo, A.olds[r] + a);
                        cp_async16(ln, A.news[r] + a);
                    } else {
                        uint4 o, n;
                        gather_bytes(A, segs, nseg, cur, x, raw, o, n);
                        *lo = o;
                        *ln = n;
                    }
                }
            }
        }
        cp_async_commit();
    };

    const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
    for (int s = 0; s < NS - 1; ++s) issue(s);
    for (int s = 0;; ++s) {
        const bool more = s < nsteps;
        const uint32_t x = uint32_t(s) * kStep + 32u * lane;   // the lane's first byte
        uint4 m0 = make_uint4(0u, 0u, 0u, 0u), m1 = m0, n0 = m0, n1 = m0;
        uint32_t z = 0;   // non-zero mask bytes (XOR) or changed units (overwrite) of the lane's 32
        if (more) {
            issue(s + NS - 1);
            cp_async_wait<NS - 1>();   // this lane's copies of step s have landed
            const int s0 = land_slot(lane, 0), s1 = land_slot(lane, 1);
            // a lane reads 16-byte slots that other lanes' copies filled
            __syncwarp();
            n0 = W.land[s % NS][1][s0];
            n1 = W.land[s % NS][1][s1];
            m0 = xor4(W.land[s % NS][0][s0], n0);
            m1 = xor4(W.land[s % NS][0][s1], n1);
            z = nz32(m0, m1);
            if (bits == 16) {
                changed += __popc((z | (z >> 1)) & 0x55555555u);
            } else if (bits == 8) {
                changed += __popc(z);
            } else {
                changed += nibbles_nz(m0.x) + nibbles_nz(m0.y) + nibbles_nz(m0.z) + nibbles_nz(m0.w) +
                           nibbles_nz(m1.x) + nibbles_nz(m1.y) + nibbles_nz(m1.z) + nibbles_nz(m1.w);
            }
            if (overwrite) z = unit_bits(z, ub);
        }
        // warp prefix of the per-lane counts: two ballots when no lane has more
        // than one
        const uint32_t c = __popc(z);
        uint32_t pre, tot, incl;
        if (__ballot_sync(kFull, c > 1) == 0) {
            const uint32_t any = __ballot_sync(kFull, c != 0);
            pre = __popc(any & lt);
            tot = __popc(any);
            incl = pre + c;
        } else {
            incl = warp_incl_sum(c, lane);
            pre = incl - c;
            tot = __shfl_sync(kFull, incl, 31);
        }
        if (overwrite) {
            // unit offsets straight to the body, values to `vals` (staged
            // until the count is known, or in place once it is)
            int r = units + int(pre);
            for (uint32_t b = z; b; b &= b - 1) {
                const uint32_t i = __ffs(b) - 1;
                if (r < ncap) {
                    const uint32_t u = (x + i) / ub;
                    *reinterpret_cast<uint16_t*>(body.a + 4 + 2 * r) = uint16_t(u);
                    vals[r * int(ub)] = uint8_t(byte_of32(n0, n1, i));
                    if (ub == 2) vals[r * 2 + 1] = uint8_t(byte_of32(n0, n1, i + 1));
                }
                ++r;
            }
            units += int(tot);
            if (!more) break;
            continue;
        }
        // events to the ring (by groups of 8 lanes when there are many, so
        // that at most kAppend new ones arrive at once), each part followed by
        // the parse of every full group; after the last step, the rest and
        // the virtual end event
        const int parts = tot > uint32_t(kAppend) ? 4 : 1;
        const int tail0 = tail;
        for (int hf = 0; hf < parts; ++hf) {
            if (more) {
                const bool mine = parts == 1 || (lane >> 3) == hf;
                const int end = tail0 + int(parts == 1 ? tot : __shfl_sync(kFull, incl, 8 * hf + 7));
                // the ring keeps the pending literals' events, or only the
                // unparsed ones once the chunk spills
                if (!spill && end - P.lit_ev > kRing) spill = true;
                if (mine) {
                    int e = tail0 + int(pre);
                    for (uint32_t b = z; b; b &= b - 1) {
                        const uint32_t i = __ffs(b) - 1;
                        W.pos[e & (kRing - 1)] = uint16_t(x + i);
                        W.val[e & (kRing - 1)] = uint8_t(byte_of32(m0, m1, i));
                        ++e;
                    }
                }
                tail = end;
                __syncwarp();
            }
            while (tail - np >= 32 || !more) {
                const int cnt = tail - np < 32 ? tail - np : 32;
                const bool fin = !more && tail - np < 32;
                if (fin && tail == 0) break;   // no change: no frame
                bool over = false;
                parse_group<Codec>(R, np, cnt, fin, raw, P, body, cap, !spill, lane, &over, &bad);
                np += cnt;
                if (__any_sync(kFull, over)) spill = true;
                if (fin) break;
            }
        }
        if (!more) break;
    }
}

// The stream loop of the common chunk (XOR, 16-byte-aligned pieces, 16- or
// 8-bit elements): the same steps, events and parse groups as stream_chunk
// with less work per step.  Landing stages rotate instead of being indexed
// modulo NS, this lane's copy and read addresses are worked out once, the
// warp looks up the piece of a step once, and the last groups are parsed
// after the loop.
template <int kBits, int NS, class Codec, class Out>
__device__ __forceinline__ void stream_fast(const EncArgs& A, WarpSmemT<NS>& W, const ChunkDesc& cd, const Seg* segs,
                                            int lane, const Out& body, uint32_t cap, uint32_t& changed, Parse& P,
                                            int& tail, int& np, bool& spill, bool& bad)
{
    const int raw = int(cd.raw_len);
    const int nseg = int(cd.src_count);
    const int nsteps = (raw + kStep - 1) / kStep;
    const RingSrc R{W.pos, W.val};
    const uint32_t lt = (1u << lane) - 1u;
    constexpr uint32_t kArr = sizeof(W.land[0][0]);     // one array of a stage (1 KiB)
    constexpr uint32_t kStage = sizeof(W.land[0]);      // old + new
    const uint32_t land0 = static_cast<uint32_t>(__cvta_generic_to_shared(&W.land[0][0][0]));
    const int slot_g0 = land_slot(int((16u * lane) >> 5), int(lane & 1));
    const int slot_g1 = land_slot(int((512u + 16u * lane) >> 5), int(lane & 1));
    const int rs0 = land_slot(lane, 0), rs1 = land_slot(lane, 1);

    int cur = 0, cur_u = 0;
    auto issue = [&](int s, uint32_t stage) {
        if (s < nsteps) {
            const uint32_t x0 = uint32_t(s) * kStep;
            while (cur_u + 1 < nseg && segs[cur_u + 1].off <= x0) ++cur_u;
            const Seg su = segs[cur_u];
            if (x0 + kStep <= su.off + su.len) {
                // the whole step inside one piece: one base address for the warp
                const uint32_t r = uint32_t(su.addr >> kShardShift);
                const uint64_t a = (su.addr & kAddrMask) + (x0 - su.off) + 16u * lane;
                const uint32_t d = land0 + stage * kStage;
                cp_async16_sa(d + 16u * slot_g0, A.olds[r] + a);
                cp_async16_sa(d + kArr + 16u * slot_g0, A.news[r] + a);
                cp_async16_sa(d + 16u * slot_g1, A.olds[r] + a + 512u);
                cp_async16_sa(d + kArr + 16u * slot_g1, A.news[r] + a + 512u);
            } else {
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    const uint32_t x = x0 + 512u * g + 16u * lane;
                    const int slot = g ? slot_g1 : slot_g0;
                    uint4* lo = &W.land[stage][0][slot];
                    uint4* ln = &W.land[stage][1][slot];
                    if (x >= uint32_t(raw)) {
                        *lo = *ln = make_uint4(0u, 0u, 0u, 0u);
                    } else {
                        while (cur + 1 < nseg && segs[cur + 1].off <= x) ++cur;
                        const Seg sg = segs[cur];
                        const uint32_t r = uint32_t(sg.addr >> kShardShift);
                        const uint64_t a = (sg.addr & kAddrMask) + (x - sg.off);
                        cp_async16(lo, A.olds[r] + a);
                        cp_async16(ln, A.news[r] + a);
                    }
                }
            }
        }
        cp_async_commit();
    };

#pragma unroll
    for (int i = 0; i < NS - 1; ++i) issue(i, uint32_t(i));   // NS - 1 steps ahead
    uint32_t st_in = NS - 1, st_out = 0;
    for (int s = 0; s < nsteps; ++s) {
        issue(s + NS - 1, st_in);
        st_in = st_in == NS - 1 ? 0u : st_in + 1;
        cp_async_wait<NS - 1>();   // this lane's copies of step s have landed
        __syncwarp();               // ... and the other lanes' (read below)
        const uint4 n0 = W.land[st_out][1][rs0], n1 = W.land[st_out][1][rs1];
        const uint4 m0 = xor4(W.land[st_out][0][rs0], n0), m1 = xor4(W.land[st_out][0][rs1], n1);
        st_out = st_out == NS - 1 ? 0u : st_out + 1;
        const uint32_t z = nz32(m0, m1);
        changed += kBits == 16 ? __popc((z | (z >> 1)) & 0x55555555u) : __popc(z);
        // warp prefix of the per-lane counts: two ballots when no lane has
        // more than one
        const uint32_t c = __popc(z);
        uint32_t pre, tot, incl;
        if (__ballot_sync(kFull, c > 1) == 0) {
            const uint32_t any = __ballot_sync(kFull, c != 0);
            pre = __popc(any & lt);
            tot = __popc(any);
            incl = pre + c;
        } else {
            incl = warp_incl_sum(c, lane);
            pre = incl - c;
            tot = __shfl_sync(kFull, incl, 31);
        }
        if (tot == 0) continue;
        const uint32_t x = uint32_t(s) * kStep + 32u * lane;   // the lane's first byte
        // events to the ring (by groups of 8 lanes when there are many, so
        // that at most kAppend new ones arrive at once), each part followed by
        // the parse of every full group
        const int parts = tot > uint32_t(kAppend) ? 4 : 1;
        const int tail0 = tail;
        for (int hf = 0; hf < parts; ++hf) {
            const int end = tail0 + int(parts == 1 ? tot : __shfl_sync(kFull, incl, 8 * hf + 7));
            // the ring keeps the pending literals' events, or only the
            // unparsed ones once the chunk spills
            if (!spill && end - P.lit_ev > kRing) spill = true;
            if (parts == 1 || (lane >> 3) == hf) {
                int e = tail0 + int(pre);
                for (uint32_t b = z; b; b &= b - 1) {
                    const uint32_t i = __ffs(b) - 1;
                    W.pos[e & (kRing - 1)] = uint16_t(x + i);
                    W.val[e & (kRing - 1)] = uint8_t(byte_of32(m0, m1, i));
                    ++e;
                }
            }
            tail = end;
            __syncwarp();
            while (tail - np >= 32) {
                bool over = false;
                parse_group<Codec>(R, np, 32, false, raw, P, body, cap, !spill, lane, &over, &bad);
                np += 32;
                if (__any_sync(kFull, over)) spill = true;
            }
        }
    }
    // the rest of the events and the virtual end event
    while (tail > 0) {
        const int cnt = tail - np < 32 ? tail - np : 32;
        const bool fin = tail - np < 32;
        bool over = false;
        parse_group<Codec>(R, np, cnt, fin, raw, P, body, cap, !spill, lane, &over, &bad);
        np += cnt;
        if (__any_sync(kFull, over)) spill = true;
        if (fin) break;
    }
}

// kOvf (ovf: this warp's overflow buffer of kOvfBytes): an XOR block that
// outgrows the slot goes on there, and at the chunk's end its rest moves to
// an exact reservation in the plan's heap; a chunk for which the heap has no
// room left is re-derived by the write pass instead (as every outgrown body
// is without kOvf).
template <int NS, class Codec, bool kOvf = false>
__device__ __forceinline__ void encode_chunk(const EncArgs& A, WarpSmemT<NS>& W, uint32_t k, int lane,
                                             uint8_t* ovf)
{
    // whether the heap has room left, read alongside the chunk's descriptor
    unsigned long long heap_top = 0;
    if constexpr (kOvf) heap_top = *reinterpret_cast<volatile unsigned long long*>(&A.sc->heap_top);
    const ChunkDesc cd = A.chunks[A.chunk_begin + k];
    const int raw = int(cd.raw_len);
    const int nseg = int(cd.src_count);
    const bool cached = nseg <= kMSegCache;
    if (cached)
        for (int i = lane; i < nseg; i += 32) W.segs[i] = A.src[cd.src_begin + i];
    __syncwarp();
    const Seg* segs = cached ? W.segs : A.src + cd.src_begin;
    const bool overwrite = (cd.flags & kResidualFlag) || A.mode == DCR_MODE_OVERWRITE_ONLY;
    const bool vec = (cd.flags & kSrcVec) != 0;
    const uint32_t ub = cd.bits == 16 ? 2u : 1u;
    // records that fit the slot and whose values fit the ring's storage
    const int ncap = int((kSlotBody - 8) / (2 + ub)) < kValStage / int(ub) ? int((kSlotBody - 8) / (2 + ub))
                                                                           : kValStage / int(ub);
    uint8_t* slot = A.slots + size_t(k) * kEncSlot;
    uint8_t* body = slot + kFrameHdr;
    uint8_t* vstage = reinterpret_cast<uint8_t*>(W.pos);   // overwrite values

    uint32_t changed = 0;
    Parse P{-1, 0ull, 0, 0, Codec::preamble(uint32_t(raw))};
    int tail = 0, np = 0, units = 0;
    bool spill = false, bad = false;
    if (!overwrite && lane == 0) {   // the block's preamble (Snappy: the chunk length)
        uint32_t o = 0;
        auto put = [&](uint32_t v) { body[o++] = uint8_t(v); };
        Codec::emit_preamble(put, uint32_t(raw));
    }
    // XOR blocks may go on past the slot, into the overflow buffer, while
    // the heap has room left
    bool deep_out = false;
    if constexpr (kOvf) deep_out = !overwrite && __shfl_sync(kFull, heap_top, 0) < A.heap_cap;
    auto run = [&](const auto& sink, uint32_t cap) {
        if (!overwrite && vec && cd.bits == 16)
            stream_fast<16, NS, Codec>(A, W, cd, segs, lane, sink, cap, changed, P, tail, np, spill, bad);
        else if (!overwrite && vec && cd.bits == 8)
            stream_fast<8, NS, Codec>(A, W, cd, segs, lane, sink, cap, changed, P, tail, np, spill, bad);
        else
            stream_chunk<NS, Codec>(A, W, cd, segs, lane, sink, cap, vstage, ncap, changed, P, tail, np, units,
                                    spill, bad);
    };
    if constexpr (kOvf) {
        if (deep_out) run(SplitSink{body, ovf, kSlotBody}, kSlotBody + kOvfBytes);
        else run(Sink{body}, kSlotBody);
    } else {
        run(Sink{body}, kSlotBody);
    }
    changed = __reduce_add_sync(kFull, changed);
    if (lane == 0 && changed) {
        atomicAdd(&A.counts[cd.tensor], (unsigned long long)changed);
        atomicAdd(reinterpret_cast<unsigned long long*>(&A.sc->changed), (unsigned long long)changed);
    }

    uint32_t kind = 0, body_len = 0;
    bool staged = false;
    if (changed && !overwrite) {
        if (P.out < uint32_t(raw)) {
            kind = Codec::kKind;
            body_len = P.out;
            staged = !spill;
        } else {
            kind = kXorRaw;
            body_len = uint32_t(raw);
        }
    } else if (changed) {
        const uint32_t pad = (4 - (2 * uint32_t(units)) % 4) % 4;
        const uint32_t rec = 4 + 2 * uint32_t(units) + pad + uint32_t(units) * ub;
        if (rec < uint32_t(raw)) {
            kind = kOverwrite;
            body_len = rec;
            staged = units <= ncap;
        } else {
            kind = kOverwriteDense;
            body_len = uint32_t(raw);
        }
    }
    if (__any_sync(kFull, bad) && lane == 0) report(A.sc, DCR_ERR_CORRUPT);
    const uint32_t fsz = kind ? (kFrameHdr + body_len + 15) / 16 * 16 : 0u;
    // a block past the slot: its rest and the frame's padding (a multiple of
    // 16 bytes) from the overflow buffer to the heap
    bool heaped = false;
    if (kOvf && kind && staged && fsz > kEncSlot) {   // (deep_out: only then can a staged body pass the slot)
        const uint32_t hl = fsz - kEncSlot, rest = body_len - kSlotBody;
        unsigned long long off = 0;
        if (lane == 0) off = atomicAdd(reinterpret_cast<unsigned long long*>(&A.sc->heap_top), (unsigned long long)hl);
        off = __shfl_sync(kFull, off, 0);
        if (off + hl <= A.heap_cap) {
            uint8_t* h = A.heap + off;
            for (uint32_t v = lane; v < hl / 16; v += 32)
                reinterpret_cast<uint4*>(h)[v] = reinterpret_cast<const uint4*>(ovf)[v];
            __syncwarp();
            for (uint32_t i = rest + lane; i < hl; i += 32) h[i] = 0;
            if (lane == 0) A.heapoff[k] = off;
            heaped = true;
        } else {
            staged = false;   // the heap is full: the write pass re-derives this body
        }
    }
    if (kind && !staged) {
        if (lane == 0) {
            A.fsize[k] = fsz | kSpilled;
            A.spill[atomicAdd(&A.sc->n_spill, 1u)] =
                SpillRec{k, kind, body_len, uint32_t(units), changed, {0u, 0u, 0u}};
        }
        return;
    }
    if (kind == kOverwrite) {
        const uint32_t nu = uint32_t(units);
        const uint32_t voff = 4 + 2 * nu + (4 - (2 * nu) % 4) % 4;
        for (uint32_t i = 4 + 2 * nu + lane; i < voff; i += 32) body[i] = 0;
        for (uint32_t i = lane; i < nu * ub; i += 32) body[voff + i] = vstage[i];
        if (lane == 0) *reinterpret_cast<uint32_t*>(body) = nu;
    }
    if (kind) {
        const uint32_t in_slot = fsz < kEncSlot ? fsz : kEncSlot;
        for (uint32_t i = kFrameHdr + body_len + lane; i < in_slot; i += 32) slot[i] = 0;   // padding
        if (lane == 0) write_header(slot, kind, cd.bits, A.chunk_begin + k, uint32_t(raw), body_len, changed);
    }
    if (lane == 0) A.fsize[k] = fsz | (heaped ? kHeap : 0u);
    __syncwarp();   // the ring and the overflow buffer are reused by the next chunk
}

template <int NS, class Codec, bool kOvf>
__global__ void __launch_bounds__(kMThreads, 4) encode_kernel(EncArgs A)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    WarpSmemT<NS>& W = reinterpret_cast<WarpSmemT<NS>*>(smem_raw)[threadIdx.x >> 5];
    for (;;) {
        uint32_t k = 0;
        if (lane == 0) {
            k = atomicAdd(&A.sc->ticket, 1u);
            if (*(volatile int32_t*)&A.sc->err) k = UINT_MAX;
        }
        k = __shfl_sync(kFull, k, 0);
        if (k >= A.chunk_count) break;
        uint8_t* ovf = kOvf ? A.ovf + size_t(blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * kOvfBytes
                            : nullptr;
        encode_chunk<NS, Codec, kOvf>(A, W, k, lane, ovf);
    }
}

// --------------------------------------------------------- restream_kernel --
// One listed chunk streamed again by one warp, once the frame offsets are
// known: the same stream loop and parse groups as encode_chunk, writing the
// body straight to its place in the stream (capacity: the size found the
// first time).  Overwrite values go to their place directly, the unit count
// being known.  Raw and dense frames, and LZ4 chunks whose pending literals
// outgrow the event ring, are listed for spill_kernel.
template <class Codec>
__device__ __forceinline__ void restream_chunk(const EncArgs& A, WarpSmem& W, uint32_t s, int lane)
{
    const SpillRec R = A.spill[s];
    if (R.kind == kXorRaw || R.kind == kOverwriteDense) {
        if (lane == 0) A.deep[atomicAdd(&A.sc->n_deep, 1u)] = s;
        return;
    }
    const ChunkDesc cd = A.chunks[A.chunk_begin + R.k];
    const int nseg = int(cd.src_count);
    const bool cached = nseg <= kMSegCache;
    if (cached)
        for (int i = lane; i < nseg; i += 32) W.segs[i] = A.src[cd.src_begin + i];
    __syncwarp();
    const Seg* segs = cached ? W.segs : A.src + cd.src_begin;
    const bool vec = (cd.flags & kSrcVec) != 0;
    uint8_t* f = A.frames + (A.lb[R.k] & kLbByteMask);
    uint8_t* body = f + kFrameHdr;
    const uint32_t nu = R.n_units;
    const uint32_t voff = 4 + 2 * nu + (4 - (2 * nu) % 4) % 4;

    uint32_t changed = 0;
    Parse P{-1, 0ull, 0, 0, R.kind == kOverwrite ? 0u : Codec::preamble(cd.raw_len)};
    int tail = 0, np = 0, units = 0;
    bool spill = false, bad = false;
    if (R.kind != kOverwrite && lane == 0) {   // the block's preamble
        uint32_t o = 0;
        auto put = [&](uint32_t v) { body[o++] = uint8_t(v); };
        Codec::emit_preamble(put, cd.raw_len);
    }
    const Sink sink{body};
    if (R.kind == kOverwrite)
        stream_chunk<kNS, Codec>(A, W, cd, segs, lane, sink, R.body_len, body + voff, int(nu), changed, P, tail, np,
                                 units, spill, bad);
    else if (vec && cd.bits == 16)
        stream_fast<16, kNS, Codec>(A, W, cd, segs, lane, sink, R.body_len, changed, P, tail, np, spill, bad);
    else if (vec && cd.bits == 8)
        stream_fast<8, kNS, Codec>(A, W, cd, segs, lane, sink, R.body_len, changed, P, tail, np, spill, bad);
    else
        stream_chunk<kNS, Codec>(A, W, cd, segs, lane, sink, R.body_len, nullptr, 0, changed, P, tail, np, units,
                                 spill, bad);
    changed = __reduce_add_sync(kFull, changed);
    if (R.kind == kOverwrite) {
        bad |= uint32_t(units) != nu;
        for (uint32_t i = 4 + 2 * nu + lane; i < voff; i += 32) body[i] = 0;
        if (lane == 0) *reinterpret_cast<uint32_t*>(body) = nu;
    } else {
        bad |= P.out != R.body_len;
    }
    bad |= changed != R.changed;
    if (__any_sync(kFull, bad)) {
        if (lane == 0) report(A.sc, DCR_ERR_CORRUPT);
        return;
    }
    if (R.kind == Codec::kKind && spill) {   // the ring could not hold the pending literals
        if (lane == 0) A.deep[atomicAdd(&A.sc->n_deep, 1u)] = s;
        return;
    }
    const uint32_t fsz = (kFrameHdr + R.body_len + 15) / 16 * 16;
    for (uint32_t i = kFrameHdr + R.body_len + lane; i < fsz; i += 32) f[i] = 0;   // padding
    if (lane == 0) write_header(f, R.kind, cd.bits, A.chunk_begin + R.k, cd.raw_len, R.body_len, R.changed);
    __syncwarp();   // the ring is reused by the next chunk
}

template <class Codec>
__global__ void __launch_bounds__(kMThreads, 4) restream_kernel(EncArgs A)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    const int lane = threadIdx.x & 31;
    WarpSmem& W = reinterpret_cast<WarpSmem*>(smem_raw)[threadIdx.x >> 5];
    const uint32_t n_spill = A.sc->n_spill;   // final: written by encode_kernel only
    if (n_spill == 0 || A.sc->total > A.cap) return;
    for (;;) {
        uint32_t s = 0;
        if (lane == 0) {
            s = atomicAdd(&A.sc->spill_ticket, 1u);
            if (*(volatile int32_t*)&A.sc->err) s = UINT_MAX;
        }
        s = __shfl_sync(kFull, s, 0);
        if (s >= n_spill) break;
        restream_chunk<Codec>(A, W, s, lane);
    }
}

// ---------------------------------------------------------- scan / copy --
// Frame offsets from the sizes, totals and the stream header.  One CTA per
// tile of kScanTile chunks, tiles taken in ticket order; a tile's offset
// comes from a decoupled look-back over the status words of the tiles
// before it (each already taken by a running CTA, since tickets go in
// order, so every wait ends; a wait that still runs past its limit, one
// second on the global timer or kScanSpin polls, reports DCR_ERR_TIMEOUT).
// The CTA of the last tile writes the totals and header.
constexpr uint32_t kScanSpin = 1u << 24;
constexpr uint64_t kScanWaitNs = 1000000000ull;

__device__ __forceinline__ uint64_t global_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint64_t ld_acquire64(const uint64_t* p)
{
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__global__ void __launch_bounds__(1024) scan_kernel(EncArgs A, uint64_t* tiles, uint64_t plan_hash, uint64_t base_v,
                                                   uint64_t target_v, uint32_t window)
{
    __shared__ unsigned long long wsum[32];
    __shared__ uint32_t s_tile;
    __shared__ unsigned long long s_excl;
    __shared__ int s_ok;
    const uint32_t n = A.chunk_count;
    const uint32_t ntiles = n ? (n + kScanTile - 1) / kScanTile : 1u;
    if (threadIdx.x == 0) s_tile = atomicAdd(&A.sc->scan_ticket, 1u);
    __syncthreads();
    const uint32_t tile = s_tile;
    if (tile >= ntiles) return;
    constexpr uint32_t per = kScanTile / 1024;
    const uint32_t b0 = tile * kScanTile + threadIdx.x * per;
    const uint32_t e = b0 + per < n ? b0 + per : (b0 < n ? n : b0);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    auto rec = [](uint32_t fs) -> unsigned long long {
        fs &= kFrameSizeMask;
        return fs ? ((1ull << kLbFrameShift) | fs) : 0ull;
    };
    uint32_t v[per];
#pragma unroll
    for (uint32_t j = 0; j < per; ++j) v[j] = b0 + j < e ? A.fsize[b0 + j] : 0u;
    unsigned long long sum = 0;
#pragma unroll
    for (uint32_t j = 0; j < per; ++j) sum += rec(v[j]);
    // block exclusive scan of the per-thread sums
    unsigned long long incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const unsigned long long o = __shfl_up_sync(kFull, incl, d);
        if (lane >= d) incl += o;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        unsigned long long w = wsum[lane], wi = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const unsigned long long o = __shfl_up_sync(kFull, wi, d);
            if (lane >= d) wi += o;
        }
        wsum[lane] = wi - w;
        if (lane == 31) {   // the tile's sum: publish it, then look back for its offset
            const unsigned long long agg = wi;
            int ok = 1;
            unsigned long long excl = 0;
            if (tile == 0) {
                if (!A.stall) atomicExch(reinterpret_cast<unsigned long long*>(&tiles[0]), kTileInc | agg);
            } else {
                atomicExch(reinterpret_cast<unsigned long long*>(&tiles[tile]), kTileAgg | agg);
                const uint64_t t0 = global_ns();
                for (int64_t j = int64_t(tile) - 1; j >= 0 && ok; --j) {
                    uint64_t s = ld_acquire64(&tiles[j]);
                    for (uint32_t spin = 0; !(s >> 62) && ok; ++spin) {
                        if (spin > kScanSpin || global_ns() - t0 > kScanWaitNs || *(volatile int32_t*)&A.sc->err)
                            ok = 0;
                        else {
                            __nanosleep(64);
                            s = ld_acquire64(&tiles[j]);
                        }
                    }
                    if (!ok) break;
                    excl += s & kTileValMask;
                    if ((s >> 62) == 2) break;
                }
                if (ok) atomicExch(reinterpret_cast<unsigned long long*>(&tiles[tile]), kTileInc | (excl + agg));
                else atomicCAS(reinterpret_cast<int*>(&A.sc->err), 0, DCR_ERR_TIMEOUT);
            }
            s_excl = excl;
            s_ok = ok;
        }
    }
    __syncthreads();
    if (!s_ok) return;
    unsigned long long run = s_excl + wsum[warp] + incl - sum;
#pragma unroll
    for (uint32_t j = 0; j < per; ++j) {
        if (b0 + j < e) A.lb[b0 + j] = run;
        run += rec(v[j]);
    }
    if (tile == ntiles - 1 && threadIdx.x == 1023) {   // run: the window's frames and bytes
        const uint64_t fbytes = run & kLbByteMask, nframes = run >> kLbFrameShift;
        const uint64_t total = kStreamHdr + fbytes + 8 * nframes;
        A.sc->total = total;
        A.sc->n_frames = nframes;
        if (A.header && total <= A.cap && !*(volatile int32_t*)&A.sc->err) {
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

// One warp per chunk: the slot's frame to its place in the stream, and the
// frame's index entry (spilled frames: the entry only).
__global__ void copy_kernel(EncArgs A)
{
    const uint64_t total = A.sc->total, nframes = A.sc->n_frames;
    if (total > A.cap || *(volatile int32_t*)&A.sc->err) return;
    uint64_t* index = A.index ? A.index : reinterpret_cast<uint64_t*>(A.payload + total - 8 * nframes);
    const int lane = threadIdx.x & 31;
    const uint32_t nw = gridDim.x * (blockDim.x >> 5);
    for (uint32_t k = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); k < A.chunk_count; k += nw) {
        const uint32_t fs = A.fsize[k];
        if (!(fs & kFrameSizeMask)) continue;
        const uint64_t ex = A.lb[k];
        const uint64_t rel = ex & kLbByteMask;
        if (lane == 0) index[ex >> kLbFrameShift] = A.frame_base + rel;
        if (fs & kSpilled) continue;
        const uint32_t size = fs & kFrameSizeMask;
        auto copy = [&](const uint4* __restrict__ src, uint4* __restrict__ dst, uint32_t nv) {
            for (uint32_t i0 = lane; i0 < nv; i0 += 128) {   // four loads in flight per lane
                uint4 v[4];
#pragma unroll
                for (uint32_t j = 0; j < 4; ++j)
                    if (i0 + 32 * j < nv) v[j] = src[i0 + 32 * j];
#pragma unroll
                for (uint32_t j = 0; j < 4; ++j)
                    if (i0 + 32 * j < nv) dst[i0 + 32 * j] = v[j];
            }
        };
        const uint32_t in_slot = size < kEncSlot ? size : kEncSlot;
        copy(reinterpret_cast<const uint4*>(A.slots + size_t(k) * kEncSlot), reinterpret_cast<uint4*>(A.frames + rel),
             in_slot / 16);
        if (fs & kHeap)   // the body's rest, from the heap
            copy(reinterpret_cast<const uint4*>(A.heap + A.heapoff[k]),
                 reinterpret_cast<uint4*>(A.frames + rel + kEncSlot), (size - kEncSlot) / 16);
    }
}

// ----------------------------------------------------------- spill_kernel --
// Gather, XOR and map one chunk's 4 KiB slice (warp w).
__device__ __forceinline__ void load_slice(const EncArgs& A, Buf& B, bool overwrite, int w, int lane)
{
    const ChunkDesc& cd = B.meta.cd;
    const int raw = int(cd.raw_len);
    const int nseg = int(cd.src_count);
    const Seg* segs = nseg <= kSegCache ? B.meta.segs : A.src + cd.src_begin;
    uint8_t* bytes = reinterpret_cast<uint8_t*>(B.data);
    const int v0 = w * kVecPerWarp;

    // bitmap word of the vector pair (v, v + 1) held by lanes (even, odd)
    auto map_vec = [&](int v, uint32_t z) {
        const uint32_t hi = __shfl_down_sync(kFull, z, 1);
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
#pragma unroll
        for (int j = 0; j < kVPL; ++j) {
            const int v = v0 + j * 32 + lane;
            const uint4 m = xor4(o[j], n[j]);
            B.data[v] = overwrite ? n[j] : m;
            map_vec(v, nz16(m));
        }
    } else {
        // unaligned pieces: byte-wise gather.  The mask is staged first;
        // overwrite chunks then restage new bytes.
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
                    map_vec(v, nz16(B.data[v]));
                }
                __syncwarp();
            }
        }
    }
}

// Appends the positions of the set bits of bitmap steps [t, ...) to B.ev
// after its first n entries, in order, until a further step might not fit.
// Returns the step reached; *n_out = entries listed in all.
__device__ __forceinline__ int list_events(Buf& B, int t, int n, int lane, int* n_out)
{
    for (; t < kSteps; ++t) {
        const uint32_t w = B.bits[32 * t + lane];
        const uint32_t c = __popc(w);
        const uint32_t incl = warp_incl_sum(c, lane);
        const uint32_t tot = __shfl_sync(kFull, incl, 31);
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

// LZ4 block of the chunk in B written to body[0, body_len); returns its size
// (body == nullptr: the size only).  Events are listed in batches; a batch's
// partial last group moves to the front of the next one, so the groups are
// those of encode_kernel.
template <class Codec>
__device__ uint32_t mask_block(Buf& B, int raw, uint8_t* body, uint32_t body_len, int lane, bool* bad)
{
    const MaskSrc S{B.ev, reinterpret_cast<const uint8_t*>(B.data)};
    Parse P{-1, 0ull, 0, 0, Codec::preamble(uint32_t(raw))};
    const bool emit = body != nullptr;
    if (emit && lane == 0) {   // the block's preamble
        uint32_t o = 0;
        auto put = [&](uint32_t v) { body[o++] = uint8_t(v); };
        Codec::emit_preamble(put, uint32_t(raw));
    }
    bool over = false;
    int t = 0, keep = 0;
    for (;;) {
        int n;
        t = list_events(B, t, keep, lane, &n);
        const bool fin = t >= kSteps;
        int g = 0;
        for (; g + 32 <= n; g += 32)
            parse_group<Codec>(S, g, 32, false, raw, P, Sink{body}, body_len, emit, lane, &over, bad);
        if (fin) {
            parse_group<Codec>(S, g, n - g, true, raw, P, Sink{body}, body_len, emit, lane, &over, bad);
            break;
        }
        const int rem = n - g;   // < 32, and g >= 32 since a batch stops only near kEvCap
        const uint16_t x = lane < rem ? B.ev[g + lane] : uint16_t(0);
        __syncwarp();
        if (lane < rem) B.ev[lane] = x;
        __syncwarp();
        keep = rem;
    }
    if (over) *bad = true;
    return P.out;
}

template <class Codec>
__global__ void __launch_bounds__(kSThreads, 2) spill_kernel(EncArgs A)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Buf& B = *reinterpret_cast<Buf*>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t n_deep = A.sc->n_deep;     // final: written by restream_kernel only
    // total: final, written by scan_kernel; after a scan that gave up, the
    // offsets of the tiles after the stalled one were never written
    if (A.sc->total > A.cap || *(volatile int32_t*)&A.sc->err) return;
    for (uint32_t i = blockIdx.x; i < n_deep; i += gridDim.x) {
        const SpillRec R = A.spill[A.deep[i]];
        const ChunkDesc cd = A.chunks[A.chunk_begin + R.k];
        if (warp == 0) {
            if (lane == 0) B.meta.cd = cd;
            const uint32_t ns = cd.src_count < uint32_t(kSegCache) ? cd.src_count : uint32_t(kSegCache);
            for (uint32_t i = lane; i < ns; i += 32) B.meta.segs[i] = A.src[cd.src_begin + i];
        }
        __syncthreads();
        const bool overwrite = (cd.flags & kResidualFlag) || A.mode == DCR_MODE_OVERWRITE_ONLY;
        load_slice(A, B, overwrite, warp, lane);
        __syncthreads();
        const int raw = int(cd.raw_len);
        const uint8_t* bytes = reinterpret_cast<const uint8_t*>(B.data);
        uint8_t* f = A.frames + (A.lb[R.k] & kLbByteMask);
        uint8_t* body = f + kFrameHdr;
        const uint32_t fsz = (kFrameHdr + R.body_len + 15) / 16 * 16;
        if (threadIdx.x == 0) write_header(f, R.kind, cd.bits, A.chunk_begin + R.k, uint32_t(raw), R.body_len, R.changed);
        if (R.kind == kXorRaw || R.kind == kOverwriteDense) {
            const int nfull = raw >> 4;
            for (int v = threadIdx.x; v < nfull; v += kSThreads) reinterpret_cast<uint4*>(body)[v] = B.data[v];
            for (int x = (nfull << 4) + threadIdx.x; x < raw; x += kSThreads) body[x] = bytes[x];
        } else if (warp == 0 && R.kind == Codec::kKind) {
            bool bad = false;
            const uint32_t got = mask_block<Codec>(B, raw, body, R.body_len, lane, &bad);
            if ((__any_sync(kFull, bad) || got != R.body_len) && lane == 0) report(A.sc, DCR_ERR_CORRUPT);
        }
        for (uint32_t x = kFrameHdr + R.body_len + threadIdx.x; x < fsz; x += kSThreads) f[x] = 0;
        __syncthreads();
    }
}

// ------------------------------------------------------- encode_cta_kernel --
// One CTA of 8 warps per chunk, for windows with fewer chunks than the GPU
// has warp slots (one warp per chunk would leave the run as long as one
// chunk's serial parse).  Each warp streams an 8 KiB slice of the chunk
// (old and new, four 16-byte vectors per lane in flight), XORs, counts the
// changed values and lists the positions and values of the slice's non-zero
// bytes in its own region of shared memory; nothing else of the chunk is
// kept.  The chunk's event e lives in the region of the warp whose events
// come before it.  The groups of 32 events are then parsed in parallel: the
// state a group carries in from the groups before it comes from three scans
// over the groups (the longest earlier zero run, the end of the last earlier
// match, the output offset), so every group is parsed exactly as the
// one-warp encoders parse it and the frames are byte-identical.  Frames that
// fit the slot are written there; raw masks and bodies over the slot are
// sized here and listed for the write pass.  Overwrite chunks, chunks whose
// pieces are not 16-byte aligned and slices with more events than their
// region holds are encoded by warp 0 with the one-warp encoder.
constexpr int kEWarps = 8;
constexpr int kEThreads = 32 * kEWarps;
constexpr int kESlice = kChunk / kEWarps;           // 8 KiB per warp
constexpr int kEVPL = kESlice / 16 / 32;            // 16 vectors per lane
constexpr int kEBatch = 2;                          // ... two at a time, the next two in flight
constexpr int kEWarpCap = 1536;                     // events a warp's region holds
constexpr int kECap = kEWarpCap * kEWarps;
constexpr int kEGroups = kECap / 32 + 1;

struct __align__(16) CtaSmem {
    union {
        struct {
            uint16_t pos[kECap];
            uint8_t val[kECap];
        } ev;
        WarpSmem w;   // warp 0's one-warp encoder
    } u;
    unsigned long long gbest[kEGroups];   // a group's longest zero run, then the longest before it
    int glit[kEGroups];                   // end of a group's last match (-1: none), then of the last before it
    int glev[kEGroups];                   // ... and the event at that end (the first pending literal event)
    uint32_t gsz[kEGroups];               // a group's bytes but its first match's sequence, then the block bytes before it
    uint32_t gm0[kEGroups];               // its first match: start << 16 | length (~0u: none)
    uint32_t goff0[kEGroups];             // ... offset, | 1 << 31 when its tail starts at the carried literal start
    uint32_t wcnt[kEWarps];               // events per slice
    uint32_t wchg[kEWarps];               // changed stored values per slice
    uint32_t base[kEWarps];               // events before each slice
    Seg segs[kMSegCache];
    uint32_t total;
};

// Events of encode_cta_kernel: event e of the chunk is entry e - base[w] of
// warp w's region, w the last warp with base[w] <= e.
struct SliceSrc {
    const uint16_t* pos;
    const uint8_t* val;
    int base[kEWarps];   // events before each slice (in registers)
    __device__ __forceinline__ int slot(int e) const
    {
        int w = 0, b = 0;
#pragma unroll
        for (int i = 1; i < kEWarps; ++i)
            if (e >= base[i]) {
                w = i;
                b = base[i];
            }
        return w * kEWarpCap + e - b;
    }
    __device__ __forceinline__ int at(int e) const { return pos[slot(e)]; }
    template <class Put>
    __device__ __forceinline__ bool lits(int a, int b, int e, int e_end, Put& put) const
    {
        for (int q = a; q < b; ++q) {
            uint32_t v = 0;
            if (e < e_end) {
                const int s = slot(e);
                if (int(pos[s]) == q) {
                    v = val[s];
                    ++e;
                }
            }
            put(v);
        }
        return e == e_end;
    }
};

// encode_cta_kernel's fallback to the one-warp encoder, out of line: the
// CTA kernel's own code stays small enough for the instruction cache
template <class Codec>
__device__ __noinline__ void encode_chunk_cold(const EncArgs& A, WarpSmem& W, uint32_t k, int lane)
{
    encode_chunk<kNS, Codec>(A, W, k, lane, nullptr);
}

template <class Codec>
__global__ void __launch_bounds__(kEThreads, 4) encode_cta_kernel(EncArgs A)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    CtaSmem& C = *reinterpret_cast<CtaSmem*>(smem_raw);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t k = blockIdx.x;
    if (k >= A.chunk_count) return;
    const ChunkDesc cd = A.chunks[A.chunk_begin + k];
    const int raw = int(cd.raw_len);
    const int nseg = int(cd.src_count);
    const bool overwrite = (cd.flags & kResidualFlag) || A.mode == DCR_MODE_OVERWRITE_ONLY;
    if (overwrite || !(cd.flags & kSrcVec)) {   // the one-warp encoder does these
        if (warp == 0) encode_chunk_cold<Codec>(A, C.u.w, k, lane);
        return;
    }
    if (nseg <= kMSegCache)
        for (int i = threadIdx.x; i < nseg; i += kEThreads) C.segs[i] = A.src[cd.src_begin + i];
    __syncthreads();
    const Seg* segs = nseg <= kMSegCache ? C.segs : A.src + cd.src_begin;

    // stream the slice: XOR, count, list the non-zero bytes in order
    uint16_t* wpos = C.u.ev.pos + warp * kEWarpCap;
    uint8_t* wval = C.u.ev.val + warp * kEWarpCap;
    const uint32_t lt = (1u << lane) - 1u;
    const int v0 = warp * (kESlice / 16);
    const int nvec = raw >> 4;
    uint32_t changed = 0, n = 0;
    int cur = 0;
    // vectors j0 .. j0 + kEBatch - 1 of this lane (zero past the chunk)
    auto load = [&](int j0, uint4* o, uint4* nw) {
#pragma unroll
        for (int j = 0; j < kEBatch; ++j) {
            const int v = v0 + (j0 + j) * 32 + lane;
            o[j] = nw[j] = make_uint4(0u, 0u, 0u, 0u);
            if (v < nvec) {
                const uint32_t x = uint32_t(v) << 4;
                while (cur + 1 < nseg && segs[cur + 1].off <= x) ++cur;
                const Seg sg = segs[cur];
                const uint32_t r = uint32_t(sg.addr >> kShardShift);
                const uint64_t a = (sg.addr & kAddrMask) + (x - sg.off);
                o[j] = ld_stream(A.olds[r] + a);
                nw[j] = ld_stream(A.news[r] + a);
            }
        }
    };
    uint4 o[kEBatch], nw[kEBatch];
    load(0, o, nw);
    for (int j0 = 0; j0 < kEVPL; j0 += kEBatch) {
        uint4 po[kEBatch], pn[kEBatch];   // the next batch, in flight while this one is listed
        if (j0 + kEBatch < kEVPL) load(j0 + kEBatch, po, pn);
#pragma unroll
        for (int j = 0; j < kEBatch; ++j) {
            const uint4 m = xor4(o[j], nw[j]);
            const uint32_t z = nz16(m);
            if (cd.bits == 16) changed += __popc((z | (z >> 1)) & 0x5555u);
            else if (cd.bits == 8) changed += __popc(z);
            else changed += nibbles_nz(m.x) + nibbles_nz(m.y) + nibbles_nz(m.z) + nibbles_nz(m.w);
            // warp prefix of the per-lane counts: two ballots when no lane has
            // more than one
            const uint32_t c = __popc(z);
            uint32_t incl, tot;
            if (__ballot_sync(kFull, c > 1) == 0) {
                const uint32_t any = __ballot_sync(kFull, c != 0);
                incl = __popc(any & lt) + c;
                tot = __popc(any);
            } else {
                incl = warp_incl_sum(c, lane);
                tot = __shfl_sync(kFull, incl, 31);
            }
            if (tot == 0) continue;
            uint32_t at = n + incl - c;
            const uint32_t x = uint32_t(v0 + (j0 + j) * 32 + lane) << 4;
            for (uint32_t b = z; b; b &= b - 1) {
                const uint32_t i = __ffs(b) - 1;
                if (at < uint32_t(kEWarpCap)) {
                    wpos[at] = uint16_t(x + i);
                    wval[at] = uint8_t(byte_of(m, i));
                }
                ++at;
            }
            n += tot;
        }
#pragma unroll
        for (int j = 0; j < kEBatch; ++j) {
            o[j] = po[j];
            nw[j] = pn[j];
        }
    }
    changed = __reduce_add_sync(kFull, changed);
    if (lane == 0) {
        C.wcnt[warp] = n;
        C.wchg[warp] = changed;
    }
    __syncthreads();
    uint32_t total_ev = 0, chunk_changed = 0;
    bool overflow = false;
#pragma unroll
    for (int w = 0; w < kEWarps; ++w) {
        const uint32_t c = C.wcnt[w];
        if (warp == 0 && lane == w) C.base[w] = total_ev;
        total_ev += c;
        chunk_changed += C.wchg[w];
        overflow |= c > uint32_t(kEWarpCap);
    }
    if (overflow) {   // a slice outgrew its region: the one-warp encoder takes the chunk
        __syncthreads();
        if (warp == 0) encode_chunk_cold<Codec>(A, C.u.w, k, lane);
        return;
    }
    if (threadIdx.x == 0 && chunk_changed) {
        atomicAdd(&A.counts[cd.tensor], (unsigned long long)chunk_changed);
        atomicAdd(reinterpret_cast<unsigned long long*>(&A.sc->changed), (unsigned long long)chunk_changed);
    }
    if (chunk_changed == 0) {
        if (threadIdx.x == 0) A.fsize[k] = 0;
        return;
    }
    __syncthreads();   // base[] written
    uint8_t* slot = A.slots + size_t(k) * kEncSlot;
    auto spill = [&](uint32_t kind, uint32_t body_len) {
        const uint32_t fsz = (kFrameHdr + body_len + 15) / 16 * 16;
        A.fsize[k] = fsz | kSpilled;
        A.spill[atomicAdd(&A.sc->n_spill, 1u)] = SpillRec{k, kind, body_len, 0u, chunk_changed, {0u, 0u, 0u}};
    };
    SliceSrc S{C.u.ev.pos, C.u.ev.val, {}};
#pragma unroll
    for (int w = 0; w < kEWarps; ++w) S.base[w] = int(C.base[w]);
    const int full = int(total_ev / 32), G = full + 1;   // full groups, then the final one (with the end event)
    auto group = [&](int g, Parse& P, uint8_t* out, uint32_t cap, bool emit, bool* over, bool* bad,
                     GroupSplit* split) {
        P.prev = g ? S.at(32 * g - 1) : -1;
        const bool fin = g == full;
        parse_group<Codec>(S, 32 * g, fin ? int(total_ev) - 32 * g : 32, fin, raw, P, Sink{out}, cap, emit, lane,
                           over, bad, split);
    };
    bool over = false, bad = false;
    // 1. each group's longest zero run (independent of the carried state):
    //    the run before each of its events (and, in the final group, before
    //    the chunk's end), as parse_group measures it, without the parse
    for (int g = warp; g < G; g += kEWarps) {
        const bool fin = g == full;
        const int total = (fin ? int(total_ev) - 32 * g : 32) + (fin ? 1 : 0);
        const bool active = lane < total;
        const int p = (!active || (fin && lane == total - 1)) ? raw : S.at(32 * g + lane);
        int pp = __shfl_up_sync(kFull, p, 1);
        if (lane == 0) pp = g ? S.at(32 * g - 1) : -1;
        const int gs = pp + 1, L = p - gs;
        const uint32_t clen = active && L > 0 ? uint32_t(L) : 0u;
        const uint32_t mlen = __reduce_max_sync(kFull, clen);
        const uint32_t mst = __reduce_max_sync(kFull, clen == mlen && mlen ? uint32_t(gs) : 0u);
        if (lane == 0) C.gbest[g] = ((unsigned long long)mlen << 32) | mst;
    }
    __syncthreads();
    if (warp == 0) {   // exclusive prefix maximum
        unsigned long long run = 0;
        for (int g0 = 0; g0 < G; g0 += 32) {
            const int g = g0 + lane;
            unsigned long long incl = g < G ? C.gbest[g] : 0ull;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const unsigned long long o = __shfl_up_sync(kFull, incl, d);
                if (lane >= d && o > incl) incl = o;
            }
            unsigned long long ex = __shfl_up_sync(kFull, incl, 1);
            if (lane == 0) ex = 0ull;
            if (ex < run) ex = run;
            if (g < G) C.gbest[g] = ex;
            const unsigned long long last = __shfl_sync(kFull, incl, 31);
            if (last > run) run = last;
        }
    }
    __syncthreads();
    // 2. each group's last match, given the longest run before it, and its
    //    bytes but those that depend on the literal start carried in
    for (int g = warp; g < G; g += kEWarps) {
        Parse P{-1, C.gbest[g], -1, 0, 0u};
        GroupSplit Sp;
        group(g, P, nullptr, 0, false, &over, &bad, &Sp);
        if (lane == 0) {
            C.glit[g] = P.lit;
            C.glev[g] = P.lit_ev;
            C.gsz[g] = Sp.indep;
            C.gm0[g] = Sp.ms0 < 0 ? ~0u : (uint32_t(Sp.ms0) << 16) | Sp.ml0;
            C.goff0[g] = Sp.off0 | (Sp.tail_dep ? 1u << 31 : 0u);
        }
    }
    __syncthreads();
    if (warp == 0) {
        // exclusive "latest match end so far", with its event (0, 0 before
        // the first); with it each group's bytes, and their exclusive prefix
        // sum after the block's preamble
        int run = 0, run_ev = 0;
        uint32_t orun = Codec::preamble(uint32_t(raw));
        for (int g0 = 0; g0 < G; g0 += 32) {
            const int g = g0 + lane;
            const int v = g < G ? C.glit[g] : -1;
            const int ve = g < G ? C.glev[g] : 0;
            const uint32_t has = __ballot_sync(kFull, v >= 0);
            const uint32_t below = has & lt;
            const int src = below ? 31 - __clz(below) : 0;
            const int from = __shfl_sync(kFull, v, src), from_ev = __shfl_sync(kFull, ve, src);
            uint32_t sz = 0;
            if (g < G) {
                const int lit_in = below ? from : run;
                C.glit[g] = lit_in;
                C.glev[g] = below ? from_ev : run_ev;
                const uint32_t m0 = C.gm0[g], o0 = C.goff0[g];
                sz = C.gsz[g];
                if (m0 != ~0u) sz += Codec::seq(uint32_t(int(m0 >> 16) - lit_in), m0 & 0xFFFFu, o0 & 0x7FFFFFFFu);
                if (o0 >> 31) sz += Codec::tail(uint32_t(raw - lit_in));
            }
            const uint32_t incl = warp_incl_sum(sz, lane);
            if (g < G) C.gsz[g] = orun + incl - sz;
            orun += __shfl_sync(kFull, incl, 31);
            if (has) {
                run = __shfl_sync(kFull, v, 31 - __clz(has));
                run_ev = __shfl_sync(kFull, ve, 31 - __clz(has));
            }
        }
        if (lane == 0) C.total = orun;
    }
    __syncthreads();
    const uint32_t total = C.total;
    if (total >= uint32_t(raw)) {
        if (threadIdx.x == 0) spill(kXorRaw, uint32_t(raw));
        return;
    }
    if (total > kSlotBody) {
        if (threadIdx.x == 0) spill(Codec::kKind, total);
        return;
    }
    // 4. the block into the slot
    uint8_t* body = slot + kFrameHdr;
    if (threadIdx.x == 0) {   // the block's preamble (Snappy: the chunk length)
        uint32_t o = 0;
        auto put = [&](uint32_t v) { body[o++] = uint8_t(v); };
        Codec::emit_preamble(put, uint32_t(raw));
    }
    for (int g = warp; g < G; g += kEWarps) {
        Parse P{-1, C.gbest[g], C.glit[g], C.glev[g], C.gsz[g]};
        group(g, P, body, kSlotBody, true, &over, &bad, nullptr);
    }
    if (__any_sync(kFull, over || bad) && lane == 0) report(A.sc, DCR_ERR_CORRUPT);
    const uint32_t fsz = (kFrameHdr + total + 15) / 16 * 16;
    for (uint32_t i = kFrameHdr + total + threadIdx.x; i < fsz; i += kEThreads) slot[i] = 0;   // padding
    if (threadIdx.x == 0) {
        write_header(slot, Codec::kKind, cd.bits, A.chunk_begin + k, uint32_t(raw), total, chunk_changed);
        A.fsize[k] = fsz;
    }
}

// ------------------------------------------------------------------ retry --
// dcr_encode_retry: the overwrite-only stream of a window built from the
// window's XOR stream and new, without old.  retry_lane_kernel: one thread
// per frame of the XOR stream checks it and claims its chunk; a ZSRC frame
// is walked in order (the one-thread walk of the apply, lane.cuh), which
// counts the changed units (16-bit words for bf16, else bytes) and changed
// stored values without materialising the mask; its frame size goes to the
// scan, and once the scan has placed every frame retry_lane_write_kernel
// walks it again and writes the records (unit offsets, new values gathered
// through the plan's sender pieces) at their place.  Frames that walk cannot
// take (raw and general blocks, matches it cannot prove) go to
// retry_kernel: one CTA per frame decodes the mask into shared memory (the
// general decoders), lists the changed units in order and gathers their new
// values:
// OVERWRITE records that fit the slot are written there; records past the
// slot, dense chunks (records not smaller than the chunk) and frames that
// already are overwrite records (copied through) are listed for
// retry_spill_kernel, which writes them at their final place once the scan
// has placed every frame.  The frames are those dcr_encode writes in
// overwrite-only mode, byte for byte.
#include "decode.cuh"
#include "lane.cuh"

constexpr int kRThreads = 256;
constexpr int kRWarps = kRThreads / 32;
constexpr uint32_t kRBusy = 1;   // frame size of a chunk being built (sizes are multiples of 16)

struct __align__(16) RSmem {
    uint4 mask[kChunk / 16];
    uint32_t wsum[kRWarps];
    Seg segs[kSegCache];
    uint32_t f, good, n, changed;
};

// exclusive prefix of v over the CTA; *total = the sum
__device__ __forceinline__ uint32_t r_excl_scan(uint32_t v, uint32_t* wsum, uint32_t* total)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const uint32_t incl = warp_incl_sum(v, lane);
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    uint32_t before = 0, tot = 0;
#pragma unroll
    for (int i = 0; i < kRWarps; ++i) {
        before += i < w ? wsum[i] : 0u;
        tot += wsum[i];
    }
    __syncthreads();
    *total = tot;
    return before + incl - v;
}

// new byte at canonical byte x of the chunk
__device__ __forceinline__ uint8_t new_byte(const EncArgs& A, const Seg* segs, int nseg, uint32_t x)
{
    const Seg sg = segs[find_seg(segs, nseg, x)];
    return A.news[uint32_t(sg.addr >> kShardShift)][(sg.addr & kAddrMask) + (x - sg.off)];
}

// The chunk's mask (in S.mask) as OVERWRITE records written to body: unit
// count, unit offsets, zero pad, new values.  Threads take contiguous ranges
// of units, so the records come out in order.
__device__ void retry_records(const EncArgs& A, RSmem& S, const ChunkDesc& cd, const Seg* segs, uint8_t* body)
{
    const uint32_t ub = cd.bits == 16 ? 2u : 1u, nu_all = cd.raw_len / ub;
    const uint32_t per = (nu_all + kRThreads - 1) / kRThreads;
    const uint32_t u0 = threadIdx.x * per, u1 = u0 + per < nu_all ? u0 + per : nu_all;
    const uint8_t* m = reinterpret_cast<const uint8_t*>(S.mask);
    auto changed_unit = [&](uint32_t u) {
        return ub == 2 ? (m[2 * u] | m[2 * u + 1]) != 0 : m[u] != 0;
    };
    uint32_t c = 0;
    for (uint32_t u = u0; u < u1; ++u) c += changed_unit(u);
    uint32_t n;
    uint32_t at = r_excl_scan(c, S.wsum, &n);
    const uint32_t voff = 4 + 2 * n + (4 - (2 * n) % 4) % 4;
    const int nseg = int(cd.src_count);
    for (uint32_t u = u0; u < u1; ++u) {
        if (!changed_unit(u)) continue;
        body[4 + 2 * at] = uint8_t(u);
        body[5 + 2 * at] = uint8_t(u >> 8);
        for (uint32_t e = 0; e < ub; ++e) body[voff + at * ub + e] = new_byte(A, segs, nseg, u * ub + e);
        ++at;
    }
    if (threadIdx.x == 0) {
        *reinterpret_cast<uint32_t*>(body) = n;
        for (uint32_t i = 4 + 2 * n; i < voff; ++i) body[i] = 0;
    }
}

// Loads the XOR stream's frame at offset fo into S: its chunk's pieces, and
// for an XOR frame the decoded mask.  Returns the frame's kind (0:
// malformed) and fills its chunk and body length.  Called by the whole CTA.
__device__ uint32_t retry_load_at(const EncArgs& A, RSmem& S, uint64_t fo, uint32_t* k_out, uint32_t* bl_out)
{
    const uint8_t* p = A.in;
    if (fo < kStreamHdr || fo % 16 || fo + kFrameHdr > A.in_idx) return 0;
    const uint4 h0 = *reinterpret_cast<const uint4*>(p + fo), h1 = *reinterpret_cast<const uint4*>(p + fo + 16);
    const uint32_t kind = h0.y & 0xFFu, fbits = (h0.y >> 8) & 0xFFu, fflags = h0.y >> 16;
    const uint32_t c = h0.z, raw = h0.w, bl = h1.x;
    if (h0.x != kFrameMagic || kind < kXorLz4 || kind > kXorSnappy || c < A.chunk_begin ||
        c >= A.chunk_begin + A.chunk_count || bl > A.in_idx - fo - kFrameHdr)
        return 0;
    const ChunkDesc cd = A.chunks[c];
    if (raw != cd.raw_len || fbits != cd.bits) return 0;
    *k_out = c - A.chunk_begin;
    *bl_out = bl;
    const uint32_t ns = cd.src_count < uint32_t(kSegCache) ? cd.src_count : uint32_t(kSegCache);
    for (uint32_t i = threadIdx.x; i < ns; i += kRThreads) S.segs[i] = A.src[cd.src_begin + i];
    if (kind == kOverwrite || kind == kOverwriteDense) {
        __syncthreads();
        return kind;
    }
    const uint8_t* body = p + fo + kFrameHdr;
    uint8_t* m = reinterpret_cast<uint8_t*>(S.mask);
    if (kind == kXorRaw) {
        if (bl != raw) return 0;
        for (uint32_t x = threadIdx.x; x < raw; x += kRThreads) m[x] = body[x];
        __syncthreads();
        return kind;
    }
    const bool zs = (fflags & kFrameZsrc) != 0;
    if (threadIdx.x < 32) {
        const bool good = kind == kXorSnappy ? warp_decode_snappy(body, bl, m, raw, zs, threadIdx.x)
                                             : warp_decode_lz4(body, bl, m, raw, zs, threadIdx.x);
        if (threadIdx.x == 0) S.good = good;
    }
    __syncthreads();
    return S.good ? kind : 0u;
}

// frame f of the XOR stream (its offset from the index)
__device__ uint32_t retry_load(const EncArgs& A, RSmem& S, uint32_t f, uint64_t* fo_out, uint32_t* k_out,
                              uint32_t* bl_out)
{
    const uint64_t fo = *reinterpret_cast<const uint64_t*>(A.in + A.in_idx + 8ull * f);
    *fo_out = fo;
    return retry_load_at(A, S, fo, k_out, bl_out);
}

// The frames retry_lane_kernel listed (checked, their chunks claimed).
__global__ void __launch_bounds__(kRThreads) retry_kernel(EncArgs A)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    RSmem& S = *reinterpret_cast<RSmem*>(smem_raw);
    const uint32_t nl = A.sc->n_deep;   // final: written by retry_lane_kernel
    for (;;) {
        if (threadIdx.x == 0) S.f = atomicAdd(&A.sc->ticket, 1u);
        __syncthreads();
        const uint32_t j = S.f;
        __syncthreads();
        if (j >= nl) break;
        uint64_t fo = 0;
        uint32_t k = 0, bl = 0;
        const uint32_t kind = retry_load(A, S, A.deep[j], &fo, &k, &bl);
        if (kind == 0) {   // a block the walk could not take, rejected by the full decode
            if (threadIdx.x == 0) report(A.sc, DCR_ERR_CORRUPT);
            __syncthreads();
            continue;
        }
        const ChunkDesc cd = A.chunks[A.chunk_begin + k];
        const Seg* segs = cd.src_count <= uint32_t(kSegCache) ? S.segs : A.src + cd.src_begin;
        uint8_t* slot = A.slots + size_t(k) * kEncSlot;
        const uint8_t* in_frame = A.in + fo;
        if (kind == kOverwrite || kind == kOverwriteDense) {   // already overwrite records: through
            const uint32_t fsz = (kFrameHdr + bl + 15) / 16 * 16;
            if (fsz <= kEncSlot) {
                for (uint32_t v = threadIdx.x; v < fsz / 16; v += kRThreads)
                    reinterpret_cast<uint4*>(slot)[v] = reinterpret_cast<const uint4*>(in_frame)[v];
                __syncthreads();
                if (threadIdx.x == 0) A.fsize[k] = fsz;
            } else if (threadIdx.x == 0) {
                A.fsize[k] = fsz | kSpilled;
                A.spill[atomicAdd(&A.sc->n_spill, 1u)] =
                    SpillRec{k, 0u, bl, 0u, 0u, {uint32_t(fo), uint32_t(fo >> 32), 0u}};   // kind 0: copy through
            }
            __syncthreads();
            continue;
        }
        // changed units and changed stored values of the mask
        const uint32_t ub = cd.bits == 16 ? 2u : 1u, raw = cd.raw_len;
        const uint8_t* m = reinterpret_cast<const uint8_t*>(S.mask);
        uint32_t units = 0, chg = 0;
        for (uint32_t u = threadIdx.x; u < raw / ub; u += kRThreads) {
            if (ub == 2) {
                units += (m[2 * u] | m[2 * u + 1]) != 0;
            } else {
                const uint32_t b = m[u];
                units += b != 0;
                chg += cd.bits == 8 ? (b != 0) : ((b & 15u) != 0) + ((b >> 4) != 0);
            }
        }
        uint32_t n, changed;
        r_excl_scan(units, S.wsum, &n);
        r_excl_scan(chg, S.wsum, &changed);
        if (ub == 2) changed = n;
        if (n == 0) {   // an XOR frame with nothing changed is not what the encoder writes
            if (threadIdx.x == 0) report(A.sc, DCR_ERR_CORRUPT);
            __syncthreads();
            continue;
        }
        const uint32_t rec = 4 + 2 * n + (4 - (2 * n) % 4) % 4 + n * ub;
        const uint32_t kind_out = rec < raw ? kOverwrite : kOverwriteDense;
        const uint32_t body_len = kind_out == kOverwrite ? rec : raw;
        const uint32_t fsz = (kFrameHdr + body_len + 15) / 16 * 16;
        if (kind_out == kOverwrite && fsz <= kEncSlot) {
            retry_records(A, S, cd, segs, slot + kFrameHdr);
            for (uint32_t i = kFrameHdr + body_len + threadIdx.x; i < fsz; i += kRThreads) slot[i] = 0;   // padding
            __syncthreads();
            if (threadIdx.x == 0) {
                write_header(slot, kOverwrite, cd.bits, A.chunk_begin + k, raw, body_len, changed);
                A.fsize[k] = fsz;
            }
        } else if (threadIdx.x == 0) {
            A.fsize[k] = fsz | kSpilled;
            A.spill[atomicAdd(&A.sc->n_spill, 1u)] =
                SpillRec{k, kind_out, body_len, n, changed, {uint32_t(fo), uint32_t(fo >> 32), 0u}};
        }
        __syncthreads();
    }
}

// The frames retry_kernel listed, at their places in the stream: frames
// copied through, dense chunks (new bytes gathered), and records past the
// slot (the mask decoded again).
__global__ void __launch_bounds__(kRThreads) retry_spill_kernel(EncArgs A)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    RSmem& S = *reinterpret_cast<RSmem*>(smem_raw);
    const uint32_t n_spill = A.sc->n_spill;   // final: written by retry_kernel only
    if (A.sc->total > A.cap || *(volatile int32_t*)&A.sc->err) return;
    for (uint32_t i = blockIdx.x; i < n_spill; i += gridDim.x) {
        const SpillRec R = A.spill[i];
        if (R.pad[2]) continue;   // records of a walked frame: retry_lane_write_kernel's
        const uint64_t fo = uint64_t(R.pad[0]) | (uint64_t(R.pad[1]) << 32);
        uint8_t* f = A.frames + (A.lb[R.k] & kLbByteMask);
        const ChunkDesc cd = A.chunks[A.chunk_begin + R.k];
        const uint32_t raw = cd.raw_len;
        if (R.kind == 0) {   // through
            const uint32_t fsz = (kFrameHdr + R.body_len + 15) / 16 * 16;
            for (uint32_t v = threadIdx.x; v < fsz / 16; v += kRThreads)
                reinterpret_cast<uint4*>(f)[v] = reinterpret_cast<const uint4*>(A.in + fo)[v];
            continue;
        }
        const uint32_t ns = cd.src_count < uint32_t(kSegCache) ? cd.src_count : uint32_t(kSegCache);
        for (uint32_t j = threadIdx.x; j < ns; j += kRThreads) S.segs[j] = A.src[cd.src_begin + j];
        __syncthreads();
        const Seg* segs = cd.src_count <= uint32_t(kSegCache) ? S.segs : A.src + cd.src_begin;
        uint8_t* body = f + kFrameHdr;
        if (R.kind == kOverwriteDense) {
            for (uint32_t x = threadIdx.x; x < raw; x += kRThreads) body[x] = new_byte(A, segs, int(cd.src_count), x);
        } else {   // the records again, from the mask decoded again (retry_kernel checked the frame)
            uint32_t k2 = 0, bl2 = 0;
            retry_load_at(A, S, fo, &k2, &bl2);
            retry_records(A, S, cd, segs, body);
        }
        const uint32_t fsz = (kFrameHdr + R.body_len + 15) / 16 * 16;
        for (uint32_t x = kFrameHdr + R.body_len + threadIdx.x; x < fsz; x += kRThreads) f[x] = 0;   // padding
        if (threadIdx.x == 0) write_header(f, R.kind, cd.bits, A.chunk_begin + R.k, raw, R.body_len, R.changed);
        __syncthreads();
    }
}

// ---- the retry's one-thread walks ----------------------------------------
constexpr int kRLThreads = 128;

// First walk: changed units (16-bit words for bf16, else bytes) and changed
// stored values (nibbles for 4-bit data) of a ZSRC frame's mask.
struct RetryCount {
    uint32_t ushift, bits, last, n, changed;
    __device__ __forceinline__ void lit(uint32_t x, uint32_t b)
    {
        const uint32_t u = x >> ushift;
        if (u != last) {
            last = u;
            ++n;
        }
        if (bits == 4) changed += ((b & 15u) != 0) + ((b >> 4) != 0);
        else changed += 1;
    }
};

// Second walk: the records' unit offsets, in order, at body + 4 (their
// new values are gathered after it, by retry_values_kernel: a gather in
// the walk would put a DRAM round trip in its chain for every unit); never
// more than the first walk's n (at counts past it, and the caller rejects
// the frame).
struct RetryWrite {
    uint8_t* body;
    uint32_t ushift, last, at, n;
    __device__ __forceinline__ void lit(uint32_t x, uint32_t)
    {
        const uint32_t u = x >> ushift;
        if (u == last) return;
        last = u;
        if (at < n) *reinterpret_cast<uint16_t*>(body + 4 + 2 * at) = uint16_t(u);
        ++at;
    }
};

// The XOR stream's frame f: checks its index entry and header as
// retry_load_at does.  0 if malformed, else its kind.
__device__ __forceinline__ uint32_t retry_frame(const EncArgs& A, uint32_t f, uint64_t* fo_out, uint32_t* k_out,
                                                uint32_t* bl_out, uint32_t* flags_out)
{
    const uint8_t* p = A.in;
    const uint64_t fo = *reinterpret_cast<const uint64_t*>(p + A.in_idx + 8ull * f);
    if (fo < kStreamHdr || fo % 16 || fo + kFrameHdr > A.in_idx) return 0;
    const uint4 h0 = *reinterpret_cast<const uint4*>(p + fo), h1 = *reinterpret_cast<const uint4*>(p + fo + 16);
    const uint32_t kind = h0.y & 0xFFu, fbits = (h0.y >> 8) & 0xFFu;
    const uint32_t c = h0.z, raw = h0.w, bl = h1.x;
    if (h0.x != kFrameMagic || kind < kXorLz4 || kind > kXorSnappy || c < A.chunk_begin ||
        c >= A.chunk_begin + A.chunk_count || bl > A.in_idx - fo - kFrameHdr)
        return 0;
    const ChunkDesc cd = A.chunks[c];
    if (raw != cd.raw_len || fbits != cd.bits) return 0;
    *fo_out = fo;
    *k_out = c - A.chunk_begin;
    *bl_out = bl;
    *flags_out = h0.y >> 16;
    return kind;
}

__global__ void __launch_bounds__(kRLThreads) retry_lane_kernel(EncArgs A)
{
    const int lane = threadIdx.x & 31;
    const uint32_t wpb = kRLThreads / 32, nw = gridDim.x * wpb;
    // 32 consecutive frames per warp, spread over the blocks first
    for (uint64_t g = uint64_t(threadIdx.x >> 5) * gridDim.x + blockIdx.x; 32 * g < A.in_frames; g += nw) {
        const uint64_t j = 32 * g + lane;
        LaneWalk<RetryCount> W;
        bool act = false;
        int res = kLStop;
        uint64_t fo = 0;
        uint32_t k = 0, bl = 0, fl = 0, kind = 0;
        bool walk = false;
        if (j < A.in_frames) {
            kind = retry_frame(A, uint32_t(j), &fo, &k, &bl, &fl);
            if (kind == 0) {
                report(A.sc, DCR_ERR_CORRUPT);
            } else if (atomicCAS(&A.fsize[k], 0u, kRBusy) != 0u) {   // a chunk has one frame
                report(A.sc, DCR_ERR_CORRUPT);
            } else if (kind == kOverwrite || kind == kOverwriteDense) {   // already records: through
                A.fsize[k] = ((kFrameHdr + bl + 15) / 16 * 16) | kSpilled;
                A.spill[atomicAdd(&A.sc->n_spill, 1u)] =
                    SpillRec{k, 0u, bl, 0u, 0u, {uint32_t(fo), uint32_t(fo >> 32), 0u}};
            } else if ((kind == kXorLz4 || kind == kXorSnappy) && (fl & kFrameZsrc)) {
                const ChunkDesc cd = A.chunks[A.chunk_begin + k];
                W.init(kind == kXorSnappy, A.in + fo + kFrameHdr, bl, cd.raw_len, 0);
                W.K = RetryCount{cd.bits == 16 ? 1u : 0u, cd.bits, 0xFFFFFFFFu, 0u, 0u};
                act = !W.sn || snappy_pre(W);
                walk = true;
            } else {
                A.deep[atomicAdd(&A.sc->n_deep, 1u)] = uint32_t(j);
            }
        }
        lane_run<false>(W, act, res);
        if (!walk) continue;
        if (res != kLValid) {   // the full decode decides
            A.deep[atomicAdd(&A.sc->n_deep, 1u)] = uint32_t(j);
            continue;
        }
        const ChunkDesc cd = A.chunks[A.chunk_begin + k];
        const uint32_t n = W.K.n, ub = cd.bits == 16 ? 2u : 1u, raw = cd.raw_len;
        const uint32_t changed = ub == 2 ? n : W.K.changed;
        if (n == 0) {   // an XOR frame with nothing changed is not what the encoder writes
            report(A.sc, DCR_ERR_CORRUPT);
            continue;
        }
        const uint32_t rec = 4 + 2 * n + (4 - (2 * n) % 4) % 4 + n * ub;
        const uint32_t kind_out = rec < raw ? kOverwrite : kOverwriteDense;
        const uint32_t body_len = kind_out == kOverwrite ? rec : raw;
        A.fsize[k] = ((kFrameHdr + body_len + 15) / 16 * 16) | kSpilled;
        // records: the second walk's (pad[2] = 1); dense: retry_spill_kernel's
        A.spill[atomicAdd(&A.sc->n_spill, 1u)] = SpillRec{
            k, kind_out, body_len, n, changed, {uint32_t(fo), uint32_t(fo >> 32), kind_out == kOverwrite ? 1u : 0u}};
    }
}

// The records of the frames retry_lane_kernel walked, at their places.
__global__ void __launch_bounds__(kRLThreads) retry_lane_write_kernel(EncArgs A)
{
    const uint32_t n_spill = A.sc->n_spill;   // final
    if (A.sc->total > A.cap || *(volatile int32_t*)&A.sc->err) return;
    const int lane = threadIdx.x & 31;
    const uint32_t wpb = kRLThreads / 32, nw = gridDim.x * wpb;
    for (uint32_t g = (threadIdx.x >> 5) * gridDim.x + blockIdx.x; 32ull * g < n_spill; g += nw) {
        const uint32_t i = 32 * g + lane;
        LaneWalk<RetryWrite> W;
        bool act = false;
        int res = kLStop;
        SpillRec R{};
        uint8_t* f = nullptr;
        if (i < n_spill) {
            R = A.spill[i];
            if (R.pad[2]) {
                const uint64_t fo = uint64_t(R.pad[0]) | (uint64_t(R.pad[1]) << 32);
                const ChunkDesc cd = A.chunks[A.chunk_begin + R.k];
                f = A.frames + (A.lb[R.k] & kLbByteMask);
                uint8_t* body = f + kFrameHdr;
                const uint32_t n = R.n_units, voff = 4 + 2 * n + (4 - (2 * n) % 4) % 4;
                *reinterpret_cast<uint32_t*>(body) = n;
                for (uint32_t x = 4 + 2 * n; x < voff; ++x) body[x] = 0;
                const uint8_t kind = A.in[fo + 4];
                W.init(kind == kXorSnappy, A.in + fo + kFrameHdr, *reinterpret_cast<const uint32_t*>(A.in + fo + 16),
                       cd.raw_len, 0);
                W.K.body = body;
                W.K.ushift = cd.bits == 16 ? 1u : 0u;
                W.K.last = 0xFFFFFFFFu;
                W.K.at = 0;
                W.K.n = n;
                act = !W.sn || snappy_pre(W);
            }
        }
        lane_run<false>(W, act, res);
        if (!f) continue;
        if (res != kLValid || W.K.at != R.n_units) {   // the first walk passed this frame
            report(A.sc, DCR_ERR_CORRUPT);
            continue;
        }
        const ChunkDesc cd = A.chunks[A.chunk_begin + R.k];
        const uint32_t fsz = (kFrameHdr + R.body_len + 15) / 16 * 16;
        for (uint32_t x = kFrameHdr + R.body_len; x < fsz; ++x) f[x] = 0;   // padding
        write_header(f, kOverwrite, cd.bits, A.chunk_begin + R.k, cd.raw_len, R.body_len, R.changed);
    }
}

// The new values of the walked frames' records: one warp per frame, a
// lane per unit (offsets written by retry_lane_write_kernel).
__global__ void __launch_bounds__(256) retry_values_kernel(EncArgs A)
{
    const uint32_t n_spill = A.sc->n_spill;   // final
    if (A.sc->total > A.cap || *(volatile int32_t*)&A.sc->err) return;
    const int lane = threadIdx.x & 31;
    const uint32_t nw = gridDim.x * (blockDim.x >> 5);
    for (uint32_t i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < n_spill; i += nw) {
        const SpillRec R = A.spill[i];
        if (!R.pad[2]) continue;
        const ChunkDesc cd = A.chunks[A.chunk_begin + R.k];
        const uint32_t ub = cd.bits == 16 ? 2u : 1u, n = R.n_units, voff = 4 + 2 * n + (4 - (2 * n) % 4) % 4;
        uint8_t* body = A.frames + (A.lb[R.k] & kLbByteMask) + kFrameHdr;
        const Seg* segs = A.src + cd.src_begin;
        for (uint32_t j = lane; j < n; j += 32) {
            const uint32_t u = *reinterpret_cast<const uint16_t*>(body + 4 + 2 * j);
            for (uint32_t e = 0; e < ub; ++e) body[voff + j * ub + e] = new_byte(A, segs, int(cd.src_count), u * ub + e);
        }
    }
}

constexpr size_t kMainSmem = sizeof(WarpSmem) * kMWarps;
constexpr size_t kDeepSmem = sizeof(WarpSmemDeep) * kDeepWarps;

}  // namespace

namespace {

// shared-memory limits of one codec's kernels
template <class Codec>
cudaError_t codec_attributes()
{
    cudaError_t e = cudaSuccess;
    for (auto f : {encode_kernel<kNS, Codec, false>, encode_kernel<kNS, Codec, true>})
        if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kMainSmem));
    for (auto f : {encode_kernel<kNSDeep, Codec, false>, encode_kernel<kNSDeep, Codec, true>})
        if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kDeepSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(restream_kernel<Codec>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(kMainSmem));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(spill_kernel<Codec>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(sizeof(Buf)));
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(encode_cta_kernel<Codec>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(sizeof(CtaSmem)));
    return e;
}

}  // namespace

int encode_kernel_config(KernelConfig* kc)
{
    {
        const cudaError_t r = cudaFuncSetAttribute(retry_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   int(sizeof(RSmem)));
        const cudaError_t r2 = r == cudaSuccess ? cudaFuncSetAttribute(retry_spill_kernel,
                                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                                       int(sizeof(RSmem)))
                                                : r;
        if (r2 != cudaSuccess) return cuda_error(r2, "retry kernel configuration");
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&kc->retry_blocks_per_sm, retry_kernel, kRThreads,
                                                          sizeof(RSmem)) != cudaSuccess ||
            kc->retry_blocks_per_sm < 1)
            kc->retry_blocks_per_sm = 1;
    }
    int dev;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&kc->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = codec_attributes<CodecLz4>();
    if (e == cudaSuccess) e = codec_attributes<CodecSnappy>();
    // residency of the LZ4 instantiations (the Snappy ones are launched with
    // the same grids: persistent CTAs that take tickets)
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&kc->enc_blocks_per_sm, encode_kernel<kNS, CodecLz4, false>,
                                                          kMThreads, kMainSmem);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&kc->enc_deep_blocks_per_sm,
                                                          encode_kernel<kNSDeep, CodecLz4, false>, 32 * kDeepWarps,
                                                          kDeepSmem);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&kc->restream_blocks_per_sm, restream_kernel<CodecLz4>,
                                                          kMThreads, kMainSmem);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&kc->spill_blocks_per_sm, spill_kernel<CodecLz4>,
                                                          kSThreads, sizeof(Buf));
    kc->enc_warps_per_block = kMWarps;
    kc->enc_deep_warps_per_block = kDeepWarps;
    if (e != cudaSuccess) return cuda_error(e, "encode kernel configuration");
    if (kc->enc_blocks_per_sm < 1 || kc->enc_deep_blocks_per_sm < 1 || kc->restream_blocks_per_sm < 1 ||
        kc->spill_blocks_per_sm < 1)
        return set_error(DCR_ERR_CUDA, "encode kernels do not fit on an SM");
    return DCR_OK;
}

namespace {

EncArgs make_args(const dcr_plan* P, uint32_t mode, uint64_t chunk_begin, uint64_t chunk_count,
                  const void* const* olds, const void* const* news)
{
    EncArgs A{};
    A.chunks = P->d_chunks;
    A.src = P->d_src;
    for (uint32_t r = 0; r < P->tp && r < DCR_MAX_TP; ++r) {
        A.olds[r] = static_cast<const uint8_t*>(olds[r]);
        A.news[r] = static_cast<const uint8_t*>(news[r]);
    }
    A.chunk_begin = uint32_t(chunk_begin);
    A.chunk_count = uint32_t(chunk_count);
    A.mode = mode;
    A.sc = static_cast<EncScratch*>(P->d_enc);
    A.counts = reinterpret_cast<unsigned long long*>(static_cast<char*>(P->d_enc) + sizeof(EncScratch));
    A.lb = P->d_lb;
    A.fsize = P->d_fsize;
    A.spill = P->d_spill;
    A.deep = P->d_deep;
    A.slots = P->d_slots;
    A.ovf = P->d_ovf;
    A.heap = P->d_heap;
    A.heap_cap = P->heap_bytes;
    A.heapoff = P->d_heapoff;
    A.stall = P->stall_scan ? 1u : 0u;
    return A;
}

// grid of the main encoder pass
unsigned main_grid(const dcr_plan* P) { return unsigned(P->kc.num_sms * P->kc.enc_blocks_per_sm); }

// The sizing pass: every chunk encoded into its slot (or sized and listed
// for the write pass), frame sizes scanned into offsets.  With a payload the
// scan also writes the stream header when the stream fits.
int launch_size(const dcr_plan* P, EncArgs& A, uint64_t plan_hash, uint64_t base_v, uint64_t target_v,
                uint32_t window, cudaStream_t s)
{
    // ticket, error, totals, spill count and per-tensor counts start at zero
    cudaError_t e = cudaMemsetAsync(P->d_enc, 0, P->enc_head_bytes, s);
    if (e != cudaSuccess) return cuda_error(e, "encode scratch reset");
    const unsigned warps = unsigned(main_grid(P) * kMWarps);
    unsigned grid = main_grid(P);
    if (warps > A.chunk_count) grid = (A.chunk_count + kMWarps - 1) / kMWarps;
    if (grid == 0) grid = 1;
    // a window of few chunks leaves most warp slots empty: then one CTA per
    // chunk (the CTA variant) is faster than one warp per chunk
    const unsigned deep_warps = unsigned(P->kc.num_sms * P->kc.enc_deep_blocks_per_sm * kDeepWarps);
    const bool cta = P->encoder == DCR_ENCODER_CTA ||
                     (P->encoder == DCR_ENCODER_AUTO && A.chunk_count <= uint32_t(P->small_window_chunks));
    const bool deep = P->encoder == DCR_ENCODER_DEEP;
    unsigned dgrid = (A.chunk_count + kDeepWarps - 1) / kDeepWarps;
    if (dgrid > deep_warps / kDeepWarps) dgrid = deep_warps / kDeepWarps;
    if (dgrid == 0) dgrid = 1;
    const bool snappy = P->codec == DCR_CODEC_SNAPPY;
    const bool ovf = P->d_ovf != nullptr && P->overflow_seen;
    if (P->profiling) cudaEventRecord(P->ev[0], s);
    const unsigned cgrid = A.chunk_count ? A.chunk_count : 1;
    if (cta && snappy)
        encode_cta_kernel<CodecSnappy><<<cgrid, kEThreads, sizeof(CtaSmem), s>>>(A);
    else if (cta)
        encode_cta_kernel<CodecLz4><<<cgrid, kEThreads, sizeof(CtaSmem), s>>>(A);
    // the overflow heap's instantiations once this plan has seen a body
    // outgrow its slot (sparse windows keep the plain stream loop)
    else if (ovf) {
        if (deep && snappy) encode_kernel<kNSDeep, CodecSnappy, true><<<dgrid, 32 * kDeepWarps, kDeepSmem, s>>>(A);
        else if (deep) encode_kernel<kNSDeep, CodecLz4, true><<<dgrid, 32 * kDeepWarps, kDeepSmem, s>>>(A);
        else if (snappy) encode_kernel<kNS, CodecSnappy, true><<<grid, kMThreads, kMainSmem, s>>>(A);
        else encode_kernel<kNS, CodecLz4, true><<<grid, kMThreads, kMainSmem, s>>>(A);
    } else if (deep && snappy)
        encode_kernel<kNSDeep, CodecSnappy, false><<<dgrid, 32 * kDeepWarps, kDeepSmem, s>>>(A);
    else if (deep)
        encode_kernel<kNSDeep, CodecLz4, false><<<dgrid, 32 * kDeepWarps, kDeepSmem, s>>>(A);
    else if (snappy)
        encode_kernel<kNS, CodecSnappy, false><<<grid, kMThreads, kMainSmem, s>>>(A);
    else
        encode_kernel<kNS, CodecLz4, false><<<grid, kMThreads, kMainSmem, s>>>(A);
    if (P->profiling) cudaEventRecord(P->ev[1], s);
    const uint32_t ntiles = A.chunk_count ? (A.chunk_count + kScanTile - 1) / kScanTile : 1u;
    e = cudaMemsetAsync(P->d_tiles, 0, ntiles * sizeof(uint64_t), s);
    if (e != cudaSuccess) return cuda_error(e, "scan tile reset");
    scan_kernel<<<ntiles, 1024, 0, s>>>(A, P->d_tiles, plan_hash, base_v, target_v, window);
    e = cudaGetLastError();
    return e == cudaSuccess ? DCR_OK : cuda_error(e, "encode launch");
}

// The write pass: slot frames copied to their places, index entries written,
// outgrown bodies re-derived into place.
int launch_write(const dcr_plan* P, EncArgs& A, cudaStream_t s)
{
    // the write pass's own tickets start at zero (it may run more than once
    // after one sizing pass)
    cudaError_t e = cudaMemsetAsync(&A.sc->spill_ticket, 0, 2 * sizeof(uint32_t), s);
    if (e != cudaSuccess) return cuda_error(e, "encode scratch reset");
    unsigned cgrid = (A.chunk_count + 7) / 8;
    if (cgrid > unsigned(P->kc.num_sms * 8)) cgrid = unsigned(P->kc.num_sms * 8);
    if (cgrid == 0) cgrid = 1;
    copy_kernel<<<cgrid, 256, 0, s>>>(A);
    unsigned rgrid = unsigned(P->kc.num_sms * P->kc.restream_blocks_per_sm);
    const unsigned mg = (A.chunk_count + kMWarps - 1) / kMWarps;
    if (rgrid > mg) rgrid = mg ? mg : 1;
    const unsigned sgrid = unsigned(P->kc.num_sms * P->kc.spill_blocks_per_sm);
    if (P->codec == DCR_CODEC_SNAPPY) {
        restream_kernel<CodecSnappy><<<rgrid, kMThreads, kMainSmem, s>>>(A);
        spill_kernel<CodecSnappy><<<sgrid, kSThreads, sizeof(Buf), s>>>(A);
    } else {
        restream_kernel<CodecLz4><<<rgrid, kMThreads, kMainSmem, s>>>(A);
        spill_kernel<CodecLz4><<<sgrid, kSThreads, sizeof(Buf), s>>>(A);
    }
    e = cudaGetLastError();
    return e == cudaSuccess ? DCR_OK : cuda_error(e, "encode launch");
}

}  // namespace

int encode_launch(const dcr_plan* P, uint32_t mode, uint32_t window, const void* const* olds,
                  const void* const* news, uint64_t base_v, uint64_t target_v, void* payload,
                  size_t cap, cudaStream_t s)
{
    EncArgs A = make_args(P, mode, P->win_start[window], P->win_start[window + 1] - P->win_start[window], olds, news);
    A.payload = static_cast<uint8_t*>(payload);
    A.cap = payload ? cap : 0;
    A.frames = A.payload ? A.payload + kStreamHdr : nullptr;
    A.frame_base = kStreamHdr;
    A.index = nullptr;
    A.header = 1;
    int rc = launch_size(P, A, P->hash, base_v, target_v, window, s);
    if (rc == DCR_OK) rc = launch_write(P, A, s);
    if (P->profiling) cudaEventRecord(P->ev[2], s);
    return rc;
}

int encode_size_launch(const dcr_plan* P, uint32_t mode, uint64_t chunk_begin, uint64_t chunk_count,
                       const void* const* olds, const void* const* news, cudaStream_t s)
{
    EncArgs A = make_args(P, mode, chunk_begin, chunk_count, olds, news);
    A.cap = 0;   // no stream: only sizes and offsets
    return launch_size(P, A, P->hash, 0, 0, 0, s);
}

int encode_write_launch(const dcr_plan* P, uint32_t mode, uint64_t chunk_begin, uint64_t chunk_count,
                        const void* const* olds, const void* const* news, uint8_t* frames, uint64_t frame_base,
                        uint64_t* index, cudaStream_t s)
{
    EncArgs A = make_args(P, mode, chunk_begin, chunk_count, olds, news);
    A.cap = ~0ull;   // the caller checked the frames buffer against the sized frame bytes
    A.frames = frames;
    A.frame_base = frame_base;
    A.index = index;
    return launch_write(P, A, s);
}

int retry_launch(const dcr_plan* P, const void* in, uint64_t in_idx, uint64_t in_frames, uint32_t window,
                 uint64_t base_v, uint64_t target_v, const void* const* news, void* payload, size_t cap,
                 cudaStream_t s)
{
    EncArgs A = make_args(P, DCR_MODE_OVERWRITE_ONLY, P->win_start[window],
                          P->win_start[window + 1] - P->win_start[window], news, news);
    A.payload = static_cast<uint8_t*>(payload);
    A.cap = payload ? cap : 0;
    A.frames = A.payload ? A.payload + kStreamHdr : nullptr;
    A.frame_base = kStreamHdr;
    A.index = nullptr;
    A.header = 1;
    A.in = static_cast<const uint8_t*>(in);
    A.in_idx = in_idx;
    A.in_frames = in_frames;
    cudaError_t e = cudaMemsetAsync(P->d_enc, 0, P->enc_head_bytes, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(P->d_fsize, 0, (A.chunk_count ? A.chunk_count : 1) * sizeof(uint32_t), s);
    const uint32_t ntiles = A.chunk_count ? (A.chunk_count + kScanTile - 1) / kScanTile : 1u;
    if (e == cudaSuccess) e = cudaMemsetAsync(P->d_tiles, 0, ntiles * sizeof(uint64_t), s);
    if (e != cudaSuccess) return cuda_error(e, "retry scratch reset");
    const unsigned rgrid = unsigned(P->kc.num_sms * P->kc.retry_blocks_per_sm);
    const unsigned lgrid = unsigned(P->kc.num_sms * 8);
    if (P->profiling) cudaEventRecord(P->ev[0], s);
    retry_lane_kernel<<<lgrid, kRLThreads, 0, s>>>(A);
    retry_kernel<<<rgrid, kRThreads, sizeof(RSmem), s>>>(A);
    if (P->profiling) cudaEventRecord(P->ev[1], s);
    scan_kernel<<<ntiles, 1024, 0, s>>>(A, P->d_tiles, P->hash, base_v, target_v, window);
    unsigned cgrid = (A.chunk_count + 7) / 8;
    if (cgrid > unsigned(P->kc.num_sms * 8)) cgrid = unsigned(P->kc.num_sms * 8);
    if (cgrid == 0) cgrid = 1;
    copy_kernel<<<cgrid, 256, 0, s>>>(A);
    retry_spill_kernel<<<rgrid, kRThreads, sizeof(RSmem), s>>>(A);
    retry_lane_write_kernel<<<lgrid, kRLThreads, 0, s>>>(A);
    retry_values_kernel<<<cgrid, 256, 0, s>>>(A);
    if (P->profiling) cudaEventRecord(P->ev[2], s);
    e = cudaGetLastError();
    return e == cudaSuccess ? DCR_OK : cuda_error(e, "retry launch");
}

}  // namespace dcr
