/*
 * Seeded synthetic weight generator (CPU twin).
 *
 * Test and benchmark infrastructure only: it produces the raw bit buffers
 * (old and new weights) that both the oracle and the CUDA path consume.  It
 * holds none of the refit method's arithmetic (no XOR masks, no counting, no
 * projection, no compression).  synth_gpu.cu is its GPU twin; the two are
 * checked equal element by element by the test suite.
 *
 * Random numbers come from one counter-based generator, SplitMix64 (Steele,
 * Lea and Flood, "Fast splittable pseudorandom number generators", OOPSLA
 * 2014), using the 64-bit finaliser constants of Vigna's reference
 * splitmix64.c.  Every value depends only on (seed, stream, purpose, index),
 * so any element of any buffer can be regenerated on its own.
 *
 * Value distributions (the workloads of the refit pages: BF16 weights with
 * about 1 % of stored values changing per step, NVFP4 expert weights with
 * 0.085 % of bytes changing):
 *   - bf16 "normal": Irwin-Hall sum of four 16-bit uniforms, centred, scaled
 *     to standard deviation 0.02 by one IEEE fp32 multiply, rounded to bf16
 *     (round to nearest even).  Integer-only up to one correctly rounded
 *     multiply, so CPU and GPU agree bit for bit.
 *   - e2m1 packed bytes: uniform random bytes (two 4-bit codes each).
 *   - e4m3 scales: 0x20 + (h & 0x1f), positive scales in a narrow range.
 * Change rules (applied to selected elements, selection iff h < threshold):
 *   - PM4:    new = (old +/- k) mod 2^16, k in 1..4             (bf16)
 *   - LOW3:   90 %: new = old ^ r, r in 1..7; 10 %: the PM4 rule (bf16)
 *   - NIBBLE: one nibble of the byte set to a different code    (e2m1)
 *   - BPM4:   new = (old +/- k) mod 2^8, k in 1..4              (e4m3)
 *   - RANDOM: every byte of new uniformly random (incompressible case)
 * Planted zeros (bf16 only): an unselected element chosen with probability
 * zthr/2^64 gets old = +0 (0x0000), new = -0 (0x8000).
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#include "synth.h"

static inline uint64_t syn_mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t syn_key(uint64_t seed, uint64_t stream, uint64_t purpose)
{
    return syn_mix64(seed ^ syn_mix64(stream ^ (purpose << 56)));
}

static inline uint64_t syn_at(uint64_t key, uint64_t i)
{
    return syn_mix64(key + (i + 1) * 0x9E3779B97F4A7C15ULL);
}

static inline uint16_t syn_bf16_normal(uint64_t r)
{
    int32_t s = (int32_t)((r & 0xFFFF) + ((r >> 16) & 0xFFFF) + ((r >> 32) & 0xFFFF) + (r >> 48));
    float x = (float)(s - 131070) * SYN_BF16_SCALE;
    uint32_t u;
    memcpy(&u, &x, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static inline uint16_t syn_pm(uint16_t v, uint64_t p, uint32_t mod_mask)
{
    uint32_t k = 1u + (uint32_t)(p & 3u);
    uint32_t r = (p & 4u) ? (uint32_t)v - k : (uint32_t)v + k;
    return (uint16_t)(r & mod_mask);
}

typedef struct { uint64_t kb, ks, kp, kz, kr; } syn_keys;

static void syn_make_keys(const syn_params* P, syn_keys* K)
{
    K->kb = syn_key(P->seed, P->stream, 0);
    K->ks = syn_key(P->seed, P->stream, 1);
    K->kp = syn_key(P->seed, P->stream, 2);
    K->kz = syn_key(P->seed, P->stream, 3);
    K->kr = syn_key(P->seed, P->stream, 4);
}

static void syn_element_k(const syn_params* P, const syn_keys* K, uint64_t i,
                          uint16_t* o_old, uint16_t* o_new)
{
    uint64_t j = P->elem_base + i;
    uint64_t hb = syn_at(K->kb, j);
    uint16_t old;
    switch (P->value_kind) {
    case SYN_VAL_BF16_NORMAL: old = syn_bf16_normal(hb); break;
    case SYN_VAL_E4M3_SCALE:  old = (uint16_t)(0x20u + (hb & 0x1Fu)); break;
    default:                  old = (uint16_t)(hb & 0xFFu); break;
    }
    uint16_t nw = old;
    int sel = syn_at(K->ks, j) < P->threshold;
    uint64_t p = syn_at(K->kp, j);
    if (P->rule == SYN_RULE_RANDOM) {
        if (P->value_kind == SYN_VAL_BF16_NORMAL) {
            uint64_t w = syn_at(K->kr, j >> 2);
            nw = (uint16_t)((w >> (16 * (j & 3))) & 0xFFFFu);
        } else {
            uint64_t w = syn_at(K->kr, j >> 3);
            nw = (uint16_t)((w >> (8 * (j & 7))) & 0xFFu);
        }
    } else if (sel) {
        switch (P->rule) {
        case SYN_RULE_PM4:  nw = syn_pm(old, p, 0xFFFFu); break;
        case SYN_RULE_BPM4: nw = syn_pm(old, p, 0xFFu); break;
        case SYN_RULE_LOW3:
            if ((p >> 32) < 429496730ULL) nw = syn_pm(old, p, 0xFFFFu);
            else nw = (uint16_t)(old ^ (1u + (uint32_t)((p & 0xFFFFu) % 7u)));
            break;
        case SYN_RULE_NIBBLE: {
            uint32_t sh = (uint32_t)(p & 1u) * 4u;
            uint32_t cur = ((uint32_t)old >> sh) & 15u;
            uint32_t nc = (cur + 1u + (uint32_t)((p >> 1) % 15u)) & 15u;
            nw = (uint16_t)((old & ~(15u << sh)) | (nc << sh));
            break;
        }
        default: break;
        }
    } else if (P->zero_threshold && syn_at(K->kz, j) < P->zero_threshold) {
        old = 0x0000u;
        nw = 0x8000u;
    }
    *o_old = old;
    *o_new = nw;
}

void syn_element(const syn_params* P, uint64_t i, uint16_t* o_old, uint16_t* o_new)
{
    syn_keys K;
    syn_make_keys(P, &K);
    syn_element_k(P, &K, i, o_old, o_new);
}

/* Fill n elements (2-byte elements when value_kind is bf16, else bytes). */
void syn_fill(const syn_params* P, uint64_t n, void* old_out, void* new_out)
{
    int two = P->value_kind == SYN_VAL_BF16_NORMAL;
    syn_keys K;
    syn_make_keys(P, &K);
    for (uint64_t i = 0; i < n; ++i) {
        uint16_t o, w;
        syn_element_k(P, &K, i, &o, &w);
        if (two) {
            if (old_out) ((uint16_t*)old_out)[i] = o;
            if (new_out) ((uint16_t*)new_out)[i] = w;
        } else {
            if (old_out) ((uint8_t*)old_out)[i] = (uint8_t)o;
            if (new_out) ((uint8_t*)new_out)[i] = (uint8_t)w;
        }
    }
}

/* Number of elements among [0, n) that the rule selects (planted zeros
 * included), computed from the selection predicates alone. */
uint64_t syn_count_selected(const syn_params* P, uint64_t n)
{
    syn_keys K;
    syn_make_keys(P, &K);
    uint64_t ks = K.ks, kz = K.kz;
    uint64_t c = 0;
    for (uint64_t i = 0; i < n; ++i) {
        uint64_t j = P->elem_base + i;
        if (syn_at(ks, j) < P->threshold) ++c;
        else if (P->zero_threshold && syn_at(kz, j) < P->zero_threshold) ++c;
    }
    return c;
}
