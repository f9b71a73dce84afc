// Seeded synthetic weight generator (GPU twin of synth.c).
//
// Test and benchmark infrastructure only: fills device buffers with the same
// values, element for element, as the CPU twin (the test suite checks this).
// It holds none of the refit method's arithmetic.  The counter-based
// generator is SplitMix64 (Steele, Lea and Flood, OOPSLA 2014) with the
// finaliser constants of Vigna's splitmix64.c; see synth.c for the value
// distributions and change rules.
#include <cstdint>
#include <cuda_runtime.h>
#include "synth.h"

namespace {

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

__host__ __device__ __forceinline__ uint64_t key_of(uint64_t seed, uint64_t stream, uint64_t purpose)
{
    return mix64(seed ^ mix64(stream ^ (purpose << 56)));
}

__device__ __forceinline__ uint64_t at(uint64_t key, uint64_t i)
{
    return mix64(key + (i + 1) * 0x9E3779B97F4A7C15ULL);
}

__device__ __forceinline__ uint16_t bf16_normal(uint64_t r)
{
    int32_t s = (int32_t)((r & 0xFFFF) + ((r >> 16) & 0xFFFF) + ((r >> 32) & 0xFFFF) + (r >> 48));
    float x = __fmul_rn((float)(s - 131070), SYN_BF16_SCALE);
    uint32_t u = __float_as_uint(x);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

__device__ __forceinline__ uint16_t pm(uint16_t v, uint64_t p, uint32_t mod_mask)
{
    uint32_t k = 1u + (uint32_t)(p & 3u);
    uint32_t r = (p & 4u) ? (uint32_t)v - k : (uint32_t)v + k;
    return (uint16_t)(r & mod_mask);
}

struct Keys { uint64_t kb, ks, kp, kz, kr; };

__global__ void fill_kernel(syn_params P, Keys K, uint64_t n, void* old_out, void* new_out)
{
    const bool two = P.value_kind == SYN_VAL_BF16_NORMAL;
    for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < n;
         i += (uint64_t)gridDim.x * blockDim.x) {
        uint64_t j = P.elem_base + i;
        uint64_t hb = at(K.kb, j);
        uint16_t old;
        if (P.value_kind == SYN_VAL_BF16_NORMAL) old = bf16_normal(hb);
        else if (P.value_kind == SYN_VAL_E4M3_SCALE) old = (uint16_t)(0x20u + (hb & 0x1Fu));
        else old = (uint16_t)(hb & 0xFFu);
        uint16_t nw = old;
        bool sel = at(K.ks, j) < P.threshold;
        uint64_t p = at(K.kp, j);
        if (P.rule == SYN_RULE_RANDOM) {
            if (two) {
                uint64_t w = at(K.kr, j >> 2);
                nw = (uint16_t)((w >> (16 * (j & 3))) & 0xFFFFu);
            } else {
                uint64_t w = at(K.kr, j >> 3);
                nw = (uint16_t)((w >> (8 * (j & 7))) & 0xFFu);
            }
        } else if (sel) {
            if (P.rule == SYN_RULE_PM4) nw = pm(old, p, 0xFFFFu);
            else if (P.rule == SYN_RULE_BPM4) nw = pm(old, p, 0xFFu);
            else if (P.rule == SYN_RULE_LOW3) {
                if ((p >> 32) < 429496730ULL) nw = pm(old, p, 0xFFFFu);
                else nw = (uint16_t)(old ^ (1u + (uint32_t)((p & 0xFFFFu) % 7u)));
            } else if (P.rule == SYN_RULE_NIBBLE) {
                uint32_t sh = (uint32_t)(p & 1u) * 4u;
                uint32_t cur = ((uint32_t)old >> sh) & 15u;
                uint32_t nc = (cur + 1u + (uint32_t)((p >> 1) % 15u)) & 15u;
                nw = (uint16_t)((old & ~(15u << sh)) | (nc << sh));
            }
        } else if (P.zero_threshold && at(K.kz, j) < P.zero_threshold) {
            old = 0x0000u;
            nw = 0x8000u;
        }
        if (two) {
            if (old_out) ((uint16_t*)old_out)[i] = old;
            if (new_out) ((uint16_t*)new_out)[i] = nw;
        } else {
            if (old_out) ((uint8_t*)old_out)[i] = (uint8_t)old;
            if (new_out) ((uint8_t*)new_out)[i] = (uint8_t)nw;
        }
    }
}

}  // namespace

extern "C" int syn_fill_gpu(const syn_params* P, uint64_t n, void* old_out, void* new_out, void* stream)
{
    if (n == 0) return 0;
    Keys K{key_of(P->seed, P->stream, 0), key_of(P->seed, P->stream, 1), key_of(P->seed, P->stream, 2),
           key_of(P->seed, P->stream, 3), key_of(P->seed, P->stream, 4)};
    uint64_t blocks = (n + 255) / 256;
    if (blocks > 152ull * 32) blocks = 152ull * 32;
    fill_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(*P, K, n, old_out, new_out);
    return cudaGetLastError() == cudaSuccess ? 0 : -1;
}
