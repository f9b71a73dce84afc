// Dense refit: every canonical byte copied from the trainer shard arenas into
// the receiver arena through the plan (the full-checkpoint transfer that the
// delta refit replaces, and how a receiver arena is first filled).
#include <cuda_runtime.h>

#include <cstdint>

#include "dcr_internal.h"

namespace dcr {
namespace {

struct DenseArgs {
    const ChunkDesc* chunks;
    const Seg* src;
    const Seg* dst;
    const uint8_t* shards[DCR_MAX_TP];
    uint8_t* target;
    uint64_t n_chunks;
};

__device__ __forceinline__ int seg_of(const Seg* s, uint32_t n, uint32_t x)
{
    int lo = 0, hi = int(n) - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (s[mid].off <= x) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__global__ void dense_kernel(DenseArgs A)
{
    for (uint64_t c = blockIdx.x; c < A.n_chunks; c += gridDim.x) {
        const ChunkDesc cd = A.chunks[c];
        const Seg* ss = A.src + cd.src_begin;
        const Seg* ds = A.dst + cd.dst_begin;
        if ((cd.flags & kSrcVec) && (cd.flags & kDstVec)) {
            for (uint32_t v = threadIdx.x; v < cd.raw_len / 16; v += blockDim.x) {
                uint32_t x = 16 * v;
                const Seg a = ss[seg_of(ss, cd.src_count, x)];
                const Seg b = ds[seg_of(ds, cd.dst_count, x)];
                const uint8_t* from = A.shards[a.addr >> kShardShift] + (a.addr & kAddrMask) + (x - a.off);
                *reinterpret_cast<uint4*>(A.target + b.addr + (x - b.off)) =
                    *reinterpret_cast<const uint4*>(from);
            }
        } else {
            for (uint32_t x = threadIdx.x; x < cd.raw_len; x += blockDim.x) {
                const Seg a = ss[seg_of(ss, cd.src_count, x)];
                const Seg b = ds[seg_of(ds, cd.dst_count, x)];
                A.target[b.addr + (x - b.off)] =
                    A.shards[a.addr >> kShardShift][(a.addr & kAddrMask) + (x - a.off)];
            }
        }
    }
}

}  // namespace

int dense_launch(const dcr_plan* P, const void* const* shards, void* target, cudaStream_t s)
{
    DenseArgs A{};
    A.chunks = P->d_chunks;
    A.src = P->d_src;
    A.dst = P->d_dst;
    for (uint32_t r = 0; r < P->tp && r < DCR_MAX_TP; ++r) A.shards[r] = static_cast<const uint8_t*>(shards[r]);
    A.target = static_cast<uint8_t*>(target);
    A.n_chunks = P->n_chunks;
    unsigned grid = unsigned(P->kc.num_sms * 8);
    if (grid > P->n_chunks) grid = unsigned(P->n_chunks);
    dense_kernel<<<grid, 256, 0, s>>>(A);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? DCR_OK : cuda_error(e, "dense refit launch");
}

}  // namespace dcr
