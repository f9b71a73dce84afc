/* Seeded synthetic weight generator: parameters shared by the CPU and GPU
 * twins (synth.c, synth_gpu.cu).  Test and benchmark infrastructure only. */
#ifndef SYNTH_H
#define SYNTH_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { SYN_VAL_BF16_NORMAL = 0, SYN_VAL_BYTES = 1, SYN_VAL_E4M3_SCALE = 2 };
enum { SYN_RULE_NONE = 0, SYN_RULE_PM4 = 1, SYN_RULE_LOW3 = 2, SYN_RULE_NIBBLE = 3,
       SYN_RULE_BPM4 = 4, SYN_RULE_RANDOM = 5 };

/* 0.02 / sqrt(4 * (65536^2 - 1) / 12), rounded to fp32. */
#define SYN_BF16_SCALE 0x1.1bc77ap-21f

typedef struct {
    uint64_t seed;
    uint64_t stream;          /* one stream per (tensor, shard) region */
    uint64_t elem_base;       /* index of element 0 within the stream */
    uint64_t threshold;       /* selected iff hash < threshold */
    uint64_t zero_threshold;  /* planted +0 -> -0 iff hash < this (0: none) */
    uint32_t value_kind;      /* SYN_VAL_* */
    uint32_t rule;            /* SYN_RULE_* */
} syn_params;

void syn_element(const syn_params* P, uint64_t i, uint16_t* o_old, uint16_t* o_new);
void syn_fill(const syn_params* P, uint64_t n, void* old_out, void* new_out);
uint64_t syn_count_selected(const syn_params* P, uint64_t n);
int syn_fill_gpu(const syn_params* P, uint64_t n, void* old_out, void* new_out, void* stream);

#ifdef __cplusplus
}
#endif
#endif
