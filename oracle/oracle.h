/*
 * CPU oracle for bit-exact delta-compressed refit.  TEST INFRASTRUCTURE ONLY:
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load it.  It shares no code, header, table or helper with the CUDA
 * library it checks.
 *
 * What it computes (NeMo-DCR paper summary and popular write-up; "GPU
 * accelerated weight teleportation" blog, section "Delta update algebra"):
 *   mask = old XOR new over the raw stored bits, changed values counted
 *   bitwise, shard data projected into canonical checkpoint coordinates,
 *   XOR masks LZ4-block (or Snappy) encoded, non-affine (fused QKV) pieces sent as
 *   overwrite records; the receiver decodes and applies in place, with
 *   per-chunk dedup and an idempotent overwrite-only retry.
 * Each function in oracle.c cites the passage it follows.
 *
 * Parity unpinned: the plan hash's serialization (which fields, in which
 * order, go into the FNV-1a 64 hash) is a format convention the pages do not
 * fix; only its FNV-1a step (orc_fnv1a64) is pinned to published reference
 * values.  The greedy encoders' payload sizes are pinned as valid LZ4 and
 * Snappy blocks that round-trip, not to a size the pages print.
 */
#ifndef DCR_ORACLE_H
#define DCR_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORC_MAX_TP 16
#define ORC_CHUNK 65536u

enum { ORC_REPLICATED = 0, ORC_SPLIT_ROWS = 1, ORC_SPLIT_COLS = 2, ORC_RESIDUAL_QKV = 3 };
enum { ORC_RECV_CANONICAL = 0, ORC_RECV_ROWGROUP = 1 };
enum { ORC_MODE_HYBRID = 0, ORC_MODE_OVERWRITE_ONLY = 1 };
enum { ORC_K_XOR_LZ4 = 1, ORC_K_XOR_RAW = 2, ORC_K_OVERWRITE = 3, ORC_K_OVERWRITE_DENSE = 4,
       ORC_K_XOR_SNAPPY = 5 };
enum { ORC_CODEC_LZ4 = 0, ORC_CODEC_SNAPPY = 1 };   /* block codec of XOR masks */
enum { ORC_OK = 0, ORC_E_INVALID = -1, ORC_E_CAPACITY = -2, ORC_E_CORRUPT = -3,
       ORC_E_VERSION = -4, ORC_E_ABORTED = -5, ORC_E_NOMEM = -7, ORC_E_INCOMPLETE = -8 };

typedef struct {
    uint32_t elem_bits;   /* 16, 8 or 4 (4: two codes per byte, low nibble first) */
    uint32_t split;       /* ORC_REPLICATED / SPLIT_ROWS / SPLIT_COLS / RESIDUAL_QKV */
    uint32_t tp;
    uint32_t q_heads, kv_heads, head_dim;   /* RESIDUAL_QKV only */
    uint64_t rows, cols;  /* canonical shape (QKV: rows = (q + 2 kv) * head_dim) */
    uint64_t shard_off[ORC_MAX_TP];
    uint32_t recv_layout, recv_group, recv_slot, pad_;
    uint64_t recv_off;
} orc_tensor;

typedef struct {
    uint64_t n_parts, n_chunks, n_windows, canonical_bytes, plan_hash;
} orc_info;

typedef struct orc_state orc_state;

/* layout */
int orc_info_get(const orc_tensor* t, uint32_t n, uint64_t window_bytes, orc_info* out);
int orc_window_range(const orc_tensor* t, uint32_t n, uint64_t window_bytes, uint32_t w,
                     uint64_t* chunk_begin, uint64_t* chunk_count);
int orc_chunk_info(const orc_tensor* t, uint32_t n, uint64_t chunk, uint32_t* part_desc,
                   uint32_t* part_sub, uint64_t* part_off, uint32_t* len);
int orc_canonical(const orc_tensor* t, uint32_t sub, const uint8_t* const* shards, uint8_t* out);
int orc_receiver_dense(const orc_tensor* t, uint32_t n, const uint8_t* const* shards,
                       uint8_t* target);

/* primitives */
void orc_xor(const uint8_t* a, const uint8_t* b, uint8_t* out, uint64_t n);
uint64_t orc_count_changed(const uint8_t* mask, uint64_t nbytes, uint32_t elem_bits);
/* FNV-1a 64 of n bytes (the step the plan hash is built from) */
uint64_t orc_fnv1a64(const uint8_t* p, uint64_t n);
uint64_t orc_lz4_encode(const uint8_t* in, uint64_t n, uint8_t* out, uint64_t cap);
int orc_lz4_decode(const uint8_t* in, uint64_t n, uint8_t* out, uint64_t raw_len, uint32_t zsrc);
uint64_t orc_snappy_encode(const uint8_t* in, uint64_t n, uint8_t* out, uint64_t cap);
int orc_snappy_decode(const uint8_t* in, uint64_t n, uint8_t* out, uint64_t raw_len, uint32_t zsrc);

/* stream */
int orc_encode(const orc_tensor* t, uint32_t n, uint64_t window_bytes,
               const uint8_t* const* old_shards, const uint8_t* const* new_shards,
               uint32_t mode, uint32_t codec, uint32_t window, uint64_t base_version,
               uint64_t target_version, uint32_t threads, uint8_t* out, uint64_t cap, uint64_t* size,
               uint64_t* changed_per_tensor);

orc_state* orc_state_new(const orc_tensor* t, uint32_t n, uint64_t window_bytes, uint64_t version);
void orc_state_free(orc_state* s);
uint64_t orc_state_version(const orc_state* s);

/* abort_at: frames with index ordinal > abort_at are skipped and frame abort_at
 * is applied only to canonical chunk bytes below split (~0: no fault).
 * dedup = 0 disables the per-chunk claim (negative control only). */
int orc_apply(const orc_tensor* t, uint32_t n, uint64_t window_bytes, orc_state* s,
              const uint8_t* payload, uint64_t size, uint8_t* target, uint32_t retry_only,
              uint64_t abort_at, uint32_t split, uint32_t dedup, uint32_t threads);

#ifdef __cplusplus
}
#endif
#endif
