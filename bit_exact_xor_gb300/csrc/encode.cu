// Sender hot path: one persistent kernel that, per 64 KiB canonical chunk,
// gathers old and new through the plan's shard->canonical pieces, forms
// mask = old XOR new in shared memory, counts changed stored values, encodes
// the chunk (LZ4 block, raw mask, overwrite records or dense overwrite) and
// writes the frame straight to its final place in the stream, found by a
// decoupled look-back over the frame sizes of earlier chunks.  A small second
// kernel writes the frame index and the stream header.
//
// Method: "GPU-accelerated weight teleportation", "Delta update algebra"
// (mask = old XOR new on raw bits) and "A strong baseline with the
// Blackwell-native DE" (LZ4 block format); NeMo-DCR paper summary, "Input and
// change detection" (bitwise compare per owner shard), "Direct Projection",
// "Residual Conversion" and "Hybrid encoding and compression" (XOR masks for
// affine changes, overwrites for residual ones).
//
// LZ4 parse.  The masks are long zero runs around sparse non-zero bytes, so
// the encoder turns every zero run of at least 4 bytes into one match and
// leaves everything else as literals.  A run is copied from the longest
// earlier zero run when that one is long enough (non-overlapping copy), else
// it keeps its first zero as a literal and copies from it with offset 1.
// Every match therefore copies zero bytes only (frame flag ZSRC), the block
// obeys the format's end rules (last 5 bytes literals, no match start in the
// last 12 bytes), and the parse needs only three block-wide scans, so all
// 512 threads of the CTA encode their own 128-byte slice in parallel.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "dcr_internal.h"

namespace dcr {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kNVec = kChunk / 16;            // 16-byte vectors per chunk
constexpr int kVPT = kNVec / kThreads;        // vectors per thread (8)
constexpr int kSegCache = 128;                // sender pieces cached in smem
constexpr uint32_t kSpinLimit = 1u << 22;     // bounded look-back wait

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

struct __align__(16) Smem {
    uint4 buf[kNVec];          // mask (XOR chunks) or new bytes (overwrite chunks)
    uint16_t nz[kNVec];        // per vector: bit i set iff mask byte i != 0
    Seg segs[kSegCache];
    int scan_i[2][kWarps];
    unsigned long long scan_u[2][kWarps];
    uint32_t red;
    uint32_t k;
    uint32_t flag;
    uint64_t frame_off;
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

// changed stored values in a 16-byte vector whose non-zero-byte mask is m
// (bf16: 16-bit words; e4m3: bytes) or whose words are w (e2m1: nibbles)
__device__ __forceinline__ uint32_t changed_in(uint32_t m, uint4 v, uint32_t bits)
{
    if (bits == 16) return __popc((m | (m >> 1)) & 0x5555u);
    if (bits == 8) return __popc(m);
    uint32_t c = 0;
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t t = w[i] | (w[i] >> 1);
        t |= t >> 2;
        c += __popc(t & 0x11111111u);
    }
    return c;
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

// ---- block-wide scans --------------------------------------------------
// zero-run summary of a byte range: first/last non-zero position and the
// longest zero run strictly between two non-zero bytes, packed (len << 32 |
// start).  first == INT_MAX marks a range without non-zero bytes.
struct RunSum {
    int first, last;
    unsigned long long best;
};

__device__ __forceinline__ RunSum combine(RunSum a, RunSum b)
{
    if (a.first == INT_MAX) return b;
    if (b.first == INT_MAX) return a;
    RunSum r;
    r.first = a.first;
    r.last = b.last;
    unsigned long long g = ((unsigned long long)(uint32_t)(b.first - a.last - 1) << 32) |
                           (uint32_t)(a.last + 1);
    r.best = a.best > b.best ? a.best : b.best;
    if (g > r.best) r.best = g;
    return r;
}

__device__ __forceinline__ RunSum shfl_up_sum(RunSum v, int d)
{
    RunSum r;
    r.first = __shfl_up_sync(0xffffffffu, v.first, d);
    r.last = __shfl_up_sync(0xffffffffu, v.last, d);
    r.best = __shfl_up_sync(0xffffffffu, v.best, d);
    return r;
}

// exclusive scan of RunSum over the block (thread order = byte order)
__device__ RunSum scan_runs(RunSum v, Smem& S)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    RunSum inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        RunSum o = shfl_up_sum(inc, d);
        if (lane >= d) inc = combine(o, inc);
    }
    RunSum exc = shfl_up_sum(inc, 1);
    if (lane == 0) exc = RunSum{INT_MAX, 0, 0ull};
    if (lane == 31) {
        S.scan_i[0][w] = inc.first;
        S.scan_i[1][w] = inc.last;
        S.scan_u[0][w] = inc.best;
    }
    __syncthreads();
    RunSum pre{INT_MAX, 0, 0ull};
    for (int k = 0; k < w; ++k) pre = combine(pre, RunSum{S.scan_i[0][k], S.scan_i[1][k], S.scan_u[0][k]});
    __syncthreads();
    return combine(pre, exc);
}

// exclusive max (of non-negative ints) over the block
__device__ int scan_max(int v, Smem& S)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc = max(inc, o);
    }
    int exc = __shfl_up_sync(0xffffffffu, inc, 1);
    if (lane == 0) exc = 0;
    if (lane == 31) S.scan_i[0][w] = inc;
    __syncthreads();
    int pre = 0;
    for (int k = 0; k < w; ++k) pre = max(pre, S.scan_i[0][k]);
    __syncthreads();
    return max(pre, exc);
}

// exclusive sum over the block; *total gets the block total
__device__ uint32_t scan_sum(uint32_t v, Smem& S, uint32_t* total)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        uint32_t o = __shfl_up_sync(0xffffffffu, inc, d);
        if (lane >= d) inc += o;
    }
    if (lane == 31) S.scan_i[0][w] = int(inc);
    __syncthreads();
    uint32_t pre = 0, tot = 0;
    for (int k = 0; k < kWarps; ++k) {
        uint32_t x = uint32_t(S.scan_i[0][k]);
        if (k < w) pre += x;
        tot += x;
    }
    __syncthreads();
    *total = tot;
    return pre + inc - v;
}

// ---- per-thread zero-run walk --------------------------------------------
// Decides, for every zero run that ends in this thread's slice, whether it
// becomes a match.  prev: last non-zero byte before the slice (-1: virtual
// non-zero before the chunk); best: longest earlier zero run (len << 32 |
// start).  Emit(ms, me, off) is called for every match in order.
template <class Emit>
__device__ __forceinline__ void walk_runs(const uint32_t bm[4], int lo, int raw, bool last_thread,
                                          int prev, unsigned long long best, Emit emit)
{
    auto gap = [&](int q) {
        int gs = prev + 1;
        int L = q - gs;
        if (L > 0) {
            int me = q < raw - 5 ? q : raw - 5;
            uint32_t blen = uint32_t(best >> 32);
            int bstart = int(uint32_t(best));
            if (me - gs >= 4 && gs <= raw - 12 && blen >= uint32_t(me - gs)) {
                emit(gs, me, gs - bstart);
            } else if (me - (gs + 1) >= 4 && gs + 1 <= raw - 12) {
                emit(gs + 1, me, 1);
            }
            unsigned long long cand = ((unsigned long long)(uint32_t)L << 32) | uint32_t(gs);
            if (cand > best) best = cand;
        }
        prev = q;
    };
#pragma unroll 1
    for (int k = 0; k < 4; ++k) {
        uint32_t b = bm[k];
        while (b) {
            int i = __ffs(b) - 1;
            b &= b - 1;
            gap(lo + 32 * k + i);
        }
    }
    if (last_thread) gap(raw);
}

// Byte writer confined to one thread's slice [p, end) of the frame body: a
// sequence that would not fit is dropped and flagged instead of written.
struct Out {
    uint8_t* o;
    uint32_t p, end;
    bool over;
    __device__ __forceinline__ void put(uint32_t b)
    {
        if (p < end) o[p] = uint8_t(b);
        else over = true;
        ++p;
    }
};

__device__ __forceinline__ void put_len(Out& w, uint32_t v)
{
    // v >= 15 was stored as 15 in the token
    v -= 15;
    while (v >= 255) {
        w.put(255);
        v -= 255;
    }
    w.put(v);
}

__device__ __forceinline__ void put_seq(Out& w, const uint8_t* mask, uint32_t lit0, uint32_t ll,
                                        uint32_t off, uint32_t ml, bool last)
{
    uint32_t mc = last ? 0u : ml - 4;
    w.put(((ll >= 15 ? 15u : ll) << 4) | (mc >= 15 ? 15u : mc));
    if (ll >= 15) put_len(w, ll);
    for (uint32_t i = 0; i < ll; ++i) w.put(mask[lit0 + i]);
    if (last) return;
    w.put(off & 0xFFu);
    w.put(off >> 8);
    if (mc >= 15) put_len(w, mc);
}

// ================================================================ kernel ==
__global__ void __launch_bounds__(kThreads, 2) encode_kernel(EncArgs A)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    Smem& S = *reinterpret_cast<Smem*>(smem_raw);
    const int t = threadIdx.x;
    uint8_t* bytes = reinterpret_cast<uint8_t*>(S.buf);

    for (;;) {
        if (t == 0) {
            uint32_t k = atomicAdd(&A.sc->ticket, 1u);
            if (*(volatile int32_t*)&A.sc->err) k = UINT32_MAX;
            S.k = k;
            S.red = 0;
        }
        __syncthreads();
        const uint32_t k = S.k;
        if (k >= A.chunk_count) break;
        const ChunkDesc cd = A.chunks[A.chunk_begin + k];
        const int raw = int(cd.raw_len);
        const bool overwrite = (cd.flags & kResidualFlag) || A.mode == DCR_MODE_OVERWRITE_ONLY;
        const Seg* segs = A.src + cd.src_begin;
        const int nseg = int(cd.src_count);
        if (nseg > 1 && nseg <= kSegCache) {
            for (int i = t; i < nseg; i += kThreads) S.segs[i] = segs[i];
            __syncthreads();
            segs = S.segs;
        }

        // ---- gather old/new through the plan, XOR, per-vector masks, counts
        uint32_t my_changed = 0;
        if (cd.flags & kSrcVec) {
            const int nvec = raw >> 4;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint4 o[kVPT / 2], n[kVPT / 2];
#pragma unroll
                for (int j = 0; j < kVPT / 2; ++j) {
                    int v = t + (h * (kVPT / 2) + j) * kThreads;
                    o[j] = n[j] = make_uint4(0, 0, 0, 0);
                    if (v < nvec) {
                        uint32_t x = uint32_t(v) << 4;
                        const Seg sg = nseg == 1 ? segs[0] : segs[find_seg(segs, nseg, x)];
                        uint32_t r = uint32_t(sg.addr >> kShardShift);
                        uint64_t a = (sg.addr & kAddrMask) + (x - sg.off);
                        o[j] = ld_stream(A.olds[r] + a);
                        n[j] = ld_stream(A.news[r] + a);
                    }
                }
#pragma unroll
                for (int j = 0; j < kVPT / 2; ++j) {
                    int v = t + (h * (kVPT / 2) + j) * kThreads;
                    uint4 m = make_uint4(o[j].x ^ n[j].x, o[j].y ^ n[j].y, o[j].z ^ n[j].z, o[j].w ^ n[j].w);
                    uint32_t z = nz16(m);
                    my_changed += changed_in(z, m, cd.bits);
                    S.buf[v] = overwrite ? n[j] : m;
                    S.nz[v] = uint16_t(z);
                }
            }
        } else {
            // unaligned pieces: byte-wise gather (layouts with odd row sizes).
            // Pass 1 stages the mask; overwrite chunks then restage new bytes.
            for (int pass = 0; pass < (overwrite ? 2 : 1); ++pass) {
                if (pass == 1) {
                    for (int v = t; v < kNVec; v += kThreads) {
                        uint4 m = S.buf[v];
                        uint32_t z = nz16(m);
                        my_changed += changed_in(z, m, cd.bits);
                        S.nz[v] = uint16_t(z);
                    }
                    __syncthreads();
                }
                for (int x = t; x < int(kChunk); x += kThreads) {
                    uint8_t ob = 0, nb = 0;
                    if (x < raw) {
                        const Seg sg = segs[find_seg(segs, nseg, uint32_t(x))];
                        uint32_t r = uint32_t(sg.addr >> kShardShift);
                        uint64_t a = (sg.addr & kAddrMask) + (uint32_t(x) - sg.off);
                        ob = A.olds[r][a];
                        nb = A.news[r][a];
                    }
                    bytes[x] = pass == 1 ? nb : uint8_t(ob ^ nb);
                }
                __syncthreads();
            }
            if (!overwrite) {
                for (int v = t; v < kNVec; v += kThreads) {
                    uint4 m = S.buf[v];
                    uint32_t z = nz16(m);
                    my_changed += changed_in(z, m, cd.bits);
                    S.nz[v] = uint16_t(z);
                }
            }
        }
        my_changed = __reduce_add_sync(0xffffffffu, my_changed);
        if ((t & 31) == 0 && my_changed) atomicAdd(&S.red, my_changed);
        __syncthreads();
        const uint32_t changed = S.red;
        if (t == 0 && changed) {
            atomicAdd(&A.counts[cd.tensor], (unsigned long long)changed);
            atomicAdd(reinterpret_cast<unsigned long long*>(&A.sc->changed), (unsigned long long)changed);
        }

        // ---- plan this chunk's frame body
        const int lo = t * 128;
        uint32_t bm[4];
        {
            uint4 z = reinterpret_cast<const uint4*>(S.nz)[t];
            bm[0] = z.x; bm[1] = z.y; bm[2] = z.z; bm[3] = z.w;
        }
        const int t_last = raw > 0 ? (raw - 1) >> 7 : 0;
        uint32_t kind = 0, body_len = 0, my_off = 0, my_first_lit = 0, n_units = 0, my_sz = 0;
        int prev_last = -1;
        unsigned long long best0 = 0ull;
        if (changed) {
            if (!overwrite) {
                // scan A: zero-run summaries (thread 0 starts after a virtual
                // non-zero byte at -1, so the leading run counts as a run)
                RunSum mine{INT_MAX, 0, 0ull};
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    uint32_t b = bm[q];
                    while (b) {
                        int i = __ffs(b) - 1;
                        b &= b - 1;
                        RunSum one{lo + 32 * q + i, lo + 32 * q + i, 0ull};
                        mine = combine(mine, one);
                    }
                }
                if (t == 0) mine = combine(RunSum{-1, -1, 0ull}, mine);
                RunSum pre = scan_runs(mine, S);
                prev_last = t == 0 ? -1 : pre.last;
                best0 = t == 0 ? 0ull : pre.best;
                // pass 1: matches of this slice -> last match end (scan C)
                int first_ms = -1, first_ml = 0, last_me = 0;
                uint32_t rest = 0;
                bool active = lo < raw;
                if (active) {
                    walk_runs(bm, lo, raw, t == t_last, prev_last, best0, [&](int ms, int me, int) {
                        if (first_ms < 0) {
                            first_ms = ms;
                            first_ml = me - ms;
                        } else {
                            rest += seq_bytes(uint32_t(ms - last_me), uint32_t(me - ms));
                        }
                        last_me = me;
                    });
                }
                int lit0 = scan_max(first_ms >= 0 ? last_me : 0, S);
                // sizes (scan D)
                uint32_t sz = 0;
                if (first_ms >= 0) sz = seq_bytes(uint32_t(first_ms - lit0), uint32_t(first_ml)) + rest;
                if (active && t == t_last) {
                    uint32_t ll = uint32_t(raw - (first_ms >= 0 ? last_me : lit0));
                    sz += 1 + ext_len(ll) + ll;
                }
                uint32_t total;
                my_off = scan_sum(sz, S, &total);
                my_sz = sz;
                my_first_lit = uint32_t(lit0);
                if (total < uint32_t(raw)) {
                    kind = kXorLz4;
                    body_len = total;
                } else {
                    kind = kXorRaw;
                    body_len = uint32_t(raw);
                }
            } else {
                const uint32_t ub = cd.bits == 16 ? 2u : 1u;
                uint32_t units = 0;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    units += ub == 2 ? __popc((bm[q] | (bm[q] >> 1)) & 0x55555555u) : __popc(bm[q]);
                uint32_t total;
                my_off = scan_sum(units, S, &total);
                n_units = total;
                uint32_t pad = (4 - (2 * total) % 4) % 4;
                uint32_t rec = 4 + 2 * total + pad + total * ub;
                if (rec < uint32_t(raw)) {
                    kind = kOverwrite;
                    body_len = rec;
                } else {
                    kind = kOverwriteDense;
                    body_len = uint32_t(raw);
                }
            }
        }
        const uint32_t fsz = changed ? (kFrameHdr + body_len + 15) / 16 * 16 : 0u;

        // ---- decoupled look-back for the frame's place in the stream
        if (t == 0) {
            uint64_t agg = fsz ? ((1ull << kLbFrameShift) | fsz) : 0ull;
            uint64_t excl = 0;
            bool ok = true;
            if (k == 0) {
                st_release(&A.lb[0], kLbInc | agg);
            } else {
                st_release(&A.lb[k], kLbAgg | agg);
                for (int64_t j = int64_t(k) - 1; j >= 0; --j) {
                    uint64_t v = ld_acquire(&A.lb[j]);
                    uint32_t spins = 0;
                    while ((v >> 62) == 0) {
                        if (++spins > kSpinLimit || *(volatile int32_t*)&A.sc->err) {
                            ok = false;
                            break;
                        }
                        __nanosleep(64);
                        v = ld_acquire(&A.lb[j]);
                    }
                    if (!ok) break;
                    excl += v & kLbValMask;
                    if ((v >> 62) == 2) break;
                }
                if (ok) st_release(&A.lb[k], kLbInc | (excl + agg));
                else atomicCAS(reinterpret_cast<int*>(&A.sc->err), 0, DCR_ERR_TIMEOUT);
            }
            A.fsize[k] = fsz;
            S.frame_off = excl & kLbByteMask;
            S.flag = ok;
        }
        __syncthreads();
        if (!S.flag) break;

        // ---- write the frame
        const uint64_t foff = kStreamHdr + S.frame_off;
        if (fsz && foff + fsz <= A.cap) {
            uint8_t* f = A.payload + foff;
            uint8_t* body = f + kFrameHdr;
            if (t == 0) {
                uint32_t h[8];
                h[0] = kFrameMagic;
                h[1] = kind | (cd.bits << 8) | ((kind == kXorLz4 ? kFrameZsrc : 0u) << 16);
                h[2] = A.chunk_begin + k;
                h[3] = uint32_t(raw);
                h[4] = body_len;
                h[5] = changed;
                h[6] = 0;
                h[7] = 0;
                reinterpret_cast<uint4*>(f)[0] = make_uint4(h[0], h[1], h[2], h[3]);
                reinterpret_cast<uint4*>(f)[1] = make_uint4(h[4], h[5], h[6], h[7]);
                for (uint32_t i = kFrameHdr + body_len; i < fsz; ++i) f[i] = 0;
            }
            if (kind == kXorLz4) {
                if (lo < raw) {
                    const uint32_t end = my_off + my_sz < body_len ? my_off + my_sz : body_len;
                    Out w{body, my_off, end, false};
                    int lit = int(my_first_lit);
                    walk_runs(bm, lo, raw, t == t_last, prev_last, best0, [&](int ms, int me, int off) {
                        put_seq(w, bytes, uint32_t(lit), uint32_t(ms - lit), uint32_t(off), uint32_t(me - ms),
                                false);
                        lit = me;
                    });
                    if (t == t_last) put_seq(w, bytes, uint32_t(lit), uint32_t(raw - lit), 0, 0, true);
                    if (w.over || w.p != my_off + my_sz)   // sizing and emission disagree
                        atomicCAS(reinterpret_cast<int*>(&A.sc->err), 0, DCR_ERR_CORRUPT);
                }
            } else if (kind == kXorRaw || kind == kOverwriteDense) {
                const int nfull = raw >> 4;
                for (int v = t; v < nfull; v += kThreads) reinterpret_cast<uint4*>(body)[v] = S.buf[v];
                for (int x = (nfull << 4) + t; x < raw; x += kThreads) body[x] = bytes[x];
            } else {
                const uint32_t ub = cd.bits == 16 ? 2u : 1u;
                const uint32_t total_units = n_units;
                if (t == 0) *reinterpret_cast<uint32_t*>(body) = total_units;
                uint32_t pad = (4 - (2 * total_units) % 4) % 4;
                uint8_t* offs = body + 4;
                uint8_t* vals = body + 4 + 2 * total_units + pad;
                if (t == 0)
                    for (uint32_t i = 0; i < pad; ++i) offs[2 * total_units + i] = 0;
                uint32_t u = my_off;
#pragma unroll 1
                for (int q = 0; q < 4; ++q) {
                    uint32_t b = bm[q];
                    if (ub == 2) b = (b | (b >> 1)) & 0x55555555u;
                    while (b) {
                        int i = __ffs(b) - 1;
                        b &= b - 1;
                        uint32_t x = uint32_t(lo + 32 * q + i);   // first byte of the unit
                        uint32_t unit = x / ub;
                        offs[2 * u] = uint8_t(unit);
                        offs[2 * u + 1] = uint8_t(unit >> 8);
                        for (uint32_t e = 0; e < ub; ++e) vals[u * ub + e] = bytes[x + e];
                        ++u;
                    }
                }
            }
        }
        __syncthreads();
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
    if (kc->enc_blocks_per_sm < 1) kc->enc_blocks_per_sm = 1;
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
