/*
 * dcr.h — bit-exact delta-compressed refit (DCR) of model weights on GB300.
 *
 * The method (NeMo-DCR paper summary, "Method"; popular write-up, sections on
 * canonical coordinates, shard owners and XOR versus overwrite; paper
 * abstract; "GPU-accelerated weight teleportation", sections "Delta update
 * algebra", "A strong baseline with the Blackwell-native DE" and "Working
 * with low-precision RL"):
 *   sender:   mask = old XOR new over the raw stored bits of every trainer
 *             shard, changed stored values counted bitwise, shard data
 *             projected into canonical checkpoint coordinates by fixed affine
 *             maps, masks LZ4-block encoded, non-affine pieces (fused QKV)
 *             sent as overwrite records;
 *   receiver: frames decoded and applied in place through a precomputed plan
 *             (XOR or overwrite), per-chunk dedup so no mask lands twice, an
 *             idempotent overwrite-only retry, and a commit that binds the new
 *             version as the base of the next delta.
 *
 * Conventions for every entry point:
 *   - Return value is a dcr_status (0 = DCR_OK, negative = error).  No call
 *     aborts, exits or traps; dcr_last_error() gives the calling thread's
 *     message for the last failure.
 *   - Device buffers are plain CUDA device pointers owned by the caller; the
 *     library never frees them.  Shard arenas, the receiver arena and the
 *     payload must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is stream-ordered; dcr_encode, dcr_apply and
 *     dcr_apply_retry end with a small device-to-host status read and a
 *     synchronisation of `stream` (dcr_apply with two when frames were
 *     deferred to its second-phase kernels), so their outputs (sizes,
 *     counts, status, version) are final when they return.
 *   - A plan's scratch (frame slots, counters) and a receiver state's
 *     scratch are shared by every call that uses them: calls on one plan, or
 *     on one receiver state, must not overlap in time.
 *
 * Wire format of a stream (one per window; little-endian):
 *   header (64 B): "DCRS", u32 format=1, u64 plan_hash, u64 base_version,
 *     u64 target_version, u32 window, u32 flags (1 = overwrite-only),
 *     u32 chunk_begin, u32 chunk_count, u64 n_frames, u64 total_bytes;
 *   frames, ascending chunk id, each 16-byte aligned: header (32 B) "DCRF",
 *     u8 kind (1 XOR_LZ4, 2 XOR_RAW, 3 OVERWRITE, 4 OVERWRITE_DENSE,
 *     5 XOR_SNAPPY), u8 elem_bits, u16 flags (1 = every match / copy
 *     copies zero bytes),
 *     u32 chunk_id, u32 raw_len, u32 body_len, u32 changed, u64 0; then the
 *     body, zero padded to 16 bytes;
 *   index: n_frames x u64 frame offsets from the stream start.
 * A chunk is 64 KiB of one canonical tensor's row-major byte space (the last
 * chunk of a tensor may be short).  A chunk with no change sends no frame.
 */
#ifndef DCR_H
#define DCR_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DCR_MAX_TP 16
#define DCR_CHUNK_BYTES 65536u
#define DCR_STREAM_HEADER_BYTES 64u
#define DCR_FRAME_HEADER_BYTES 32u
#define DCR_NO_FAULT UINT64_MAX

typedef enum {
    DCR_OK = 0,
    DCR_ERR_INVALID = -1,    /* bad argument, descriptor, plan/stream mismatch */
    DCR_ERR_CAPACITY = -2,   /* payload buffer too small; *payload_size = required */
    DCR_ERR_CORRUPT = -3,    /* malformed stream or frame */
    DCR_ERR_VERSION = -4,    /* stream base_version != receiver version */
    DCR_ERR_ABORTED = -5,    /* injected fault stopped the apply part way */
    DCR_ERR_CUDA = -6,       /* a CUDA runtime call failed */
    DCR_ERR_NOMEM = -7,      /* host or device allocation failed */
    DCR_ERR_INCOMPLETE = -8, /* some framed chunks are not DONE: retry needed */
    DCR_ERR_TIMEOUT = -9     /* a bounded device wait gave up */
} dcr_status;

/* How a trainer holds a tensor (paper summary, "Direct Projection"; popular
 * write-up on fused Q/K/V). */
enum {
    DCR_REPLICATED = 0,   /* every rank holds it whole; shard 0 owns it */
    DCR_SPLIT_ROWS = 1,   /* column-parallel: dim 0 split into tp equal parts */
    DCR_SPLIT_COLS = 2,   /* row-parallel: dim 1 split into tp equal parts */
    DCR_RESIDUAL_QKV_INTERLEAVED = 3 /* fused QKV, per-shard kv groups of
                                        [q heads | k head | v head] rows;
                                        sent as overwrite records */
};

/* How the receiver stores it in its arena (blog, "Working with low-precision
 * RL"). */
enum {
    DCR_LAYOUT_CANONICAL = 0,        /* row-major canonical bytes */
    DCR_LAYOUT_ROWGROUP_INTERLEAVE = 1 /* fused pair: canonical row r goes to
                                          row (r/g)*2g + slot*g + r%g */
};

enum { DCR_MODE_HYBRID = 0, DCR_MODE_OVERWRITE_ONLY = 1 };
/* Encoder kernel variant (dcr_plan_opts.encoder); all produce the same
 * frames.  WIDE: one warp per chunk, many warps per SM, three landing stages
 * each; DEEP: one warp per chunk, fewer warps with twelve landing stages;
 * CTA: one 16-warp CTA per chunk (parallel gather, listing and parse),
 * faster when a window has fewer chunks than the GPU has warp slots; AUTO
 * picks WIDE or CTA by window size. */
enum { DCR_ENCODER_AUTO = 0, DCR_ENCODER_WIDE = 1, DCR_ENCODER_DEEP = 2, DCR_ENCODER_CTA = 3 };
/* Apply kernel variant (dcr_plan_opts.apply); all apply the same bytes.
 * WARP: one warp per frame; CTA: one 256-thread CTA per frame (parallel
 * sequence walk by pointer doubling), faster when windows have fewer frames
 * than the GPU has warp slots; LANE: one warp per frame for raw and
 * overwrite frames, one thread per ZSRC LZ4 or Snappy frame (a serial walk
 * that writes only the non-zero literal bytes: a tenth of the instructions,
 * so the fastest once a stream has tens of thousands of frames).  AUTO picks
 * CTA for plans with small windows, else WARP, and LANE for the streams with
 * about four frames or more per warp slot of the bitmap walk.  SPLIT: one
 * warp per raw and overwrite frame, and one warp per ZSRC LZ4 or Snappy
 * frame whose lanes walk 32 stretches of the body at once and join them
 * (bodies up to 6 KiB; the windowed walk above that).  Plans of the Snappy
 * codec take that walk for their ZSRC Snappy frames in every variant but
 * LANE and CTA. */
enum { DCR_APPLY_AUTO = 0, DCR_APPLY_WARP = 1, DCR_APPLY_CTA = 2, DCR_APPLY_LANE = 3, DCR_APPLY_SPLIT = 4 };
/* Block codec of XOR masks (dcr_plan_opts.codec).  LZ4 (frame kind 1) is the
 * default; Snappy (frame kind 5) is the other byte-oriented LZ77 codec the
 * method's pages compare it with (blog, "A strong baseline with the
 * Blackwell-native DE"): its copies cover at most 64 bytes, so long zero
 * runs cost more.  Every receiver decodes both. */
enum { DCR_CODEC_LZ4 = 0, DCR_CODEC_SNAPPY = 1 };

typedef struct dcr_plan dcr_plan;             /* opaque, library owned */
typedef struct dcr_recv_state dcr_recv_state; /* opaque, library owned */

/* One tensor of the model, read by dcr_plan_build only (caller owned).
 * elem_bits: 16 (bf16), 8 (e4m3 scales) or 4 (e2m1, two per byte, low
 * nibble first).  Canonical shape [rows, cols] row-major; for a fused QKV,
 * rows = (q_heads + 2 kv_heads) * head_dim and the canonical tensors are
 * q_proj, k_proj, v_proj, stored at recv_offset in that order.
 * shard_offset[r]: byte offset of shard r's local block in trainer arena r
 * (local blocks are row-major [rows/tp, cols], [rows, cols/tp] or the fused
 * QKV rows).  recv_offset: byte offset in the receiver arena (for a row-group
 * pair, both tensors give the fused tensor's offset and slot 0 or 1). */
typedef struct {
    const char* name;
    uint32_t elem_bits;
    uint32_t split;
    uint32_t tp;
    uint32_t q_heads, kv_heads, head_dim;
    uint64_t rows, cols;
    uint64_t shard_offset[DCR_MAX_TP];
    uint32_t recv_layout, recv_group, recv_slot, reserved;
    uint64_t recv_offset;
} dcr_tensor_desc;

/* dcr_plan_opts.flags.  HOST_ONLY: build the layout, windows, plan hash and
 * ownership parts on the host only, with no CUDA call (a plan for
 * dcr_plan_info_get, dcr_window_info_get, dcr_part_info_get and
 * dcr_stream_header, e.g. on a rank or process without a GPU); every call
 * that runs kernels returns DCR_ERR_INVALID for it. */
#define DCR_PLAN_HOST_ONLY 1u
/* Test only: the encoder's offset scan (one CTA per tile of 8192 chunks,
 * each waiting, with a bounded wait, for the running totals of the tiles
 * before it) runs with tile 0 never publishing its total, so in a window of
 * more than 8192 chunks every later tile's wait runs out: dcr_encode,
 * dcr_encode_part and dcr_encode_retry return DCR_ERR_TIMEOUT after about a
 * second and write no stream byte.  A window of one tile is unaffected. */
#define DCR_PLAN_TEST_STALL_SCAN 2u
#define DCR_NO_OVERFLOW 0xFFFFFFFFu

typedef struct {
    uint64_t window_bytes;   /* 0 = 16 GiB.  Windows pack whole tensors in
                                order; a tensor larger than a window is cut at
                                chunk boundaries.  At most 256 GiB. */
    uint32_t encoder;        /* DCR_ENCODER_AUTO (0), _WIDE, _DEEP or _CTA */
    uint32_t codec;          /* DCR_CODEC_LZ4 (0) or DCR_CODEC_SNAPPY */
    uint32_t flags;          /* 0, DCR_PLAN_HOST_ONLY, DCR_PLAN_TEST_STALL_SCAN */
    uint32_t apply;          /* DCR_APPLY_AUTO (0), _WARP, _CTA, _LANE or _SPLIT */
    uint32_t overflow_kib;    /* device heap for XOR blocks that outgrow their
                                6 KiB frame slot (masks of a few percent
                                change and more): 0 = one eighth of
                                the window size; DCR_NO_OVERFLOW = none (such
                                blocks are derived again from old and new by
                                a second pass, as they are once the heap is
                                full); in KiB.  With a heap the plan also holds one
                                64 KiB overflow buffer per encoder warp
                                (about 228 MiB on GB300). */
    uint32_t reserved;
} dcr_plan_opts;

typedef struct {
    uint64_t n_tensors, n_parts, n_chunks, n_windows;
    uint64_t canonical_bytes;   /* N: weight bytes of one version */
    uint64_t plan_hash;         /* FNV-1a 64 of the canonical description */
    uint64_t recv_bytes;        /* smallest receiver arena that fits */
    uint64_t shard_bytes[DCR_MAX_TP]; /* smallest trainer arenas that fit */
    uint32_t tp;
    uint32_t reserved;
} dcr_plan_info;

typedef struct {
    uint64_t chunk_begin, chunk_count;
    uint64_t canonical_bytes;   /* weight bytes in this window */
    uint64_t payload_bound;     /* worst-case stream size for this window */
} dcr_window_info;

/* Test-only fault injection for dcr_apply: frames whose index ordinal is
 * greater than abort_after_frames are skipped, and frame abort_after_frames
 * is applied only to canonical chunk bytes below abort_split and left
 * unfinished.  DCR_NO_FAULT disables it. */
typedef struct {
    uint64_t abort_after_frames;
    uint32_t abort_split;
    uint32_t reserved;
} dcr_fault;

typedef struct {
    uint64_t target_version;  /* from the stream header */
    uint64_t n_frames;        /* frames listed in the index */
    uint64_t frames_applied;  /* frames whose bytes were applied */
    uint64_t frames_skipped;  /* XOR frames skipped by dedup */
    uint64_t pending;         /* framed chunks not DONE after the call */
    uint32_t window;
    uint32_t committed;       /* 1 if this call committed target_version */
} dcr_apply_result;

/* Text of the calling thread's last error (never NULL). */
const char* dcr_last_error(void);

/* Plan build (blog, "A strong baseline with the Blackwell-native DE": tiling
 * and address metadata prepared on the host, read by the apply kernel;
 * paper summary, "Direct Projection" and "Residual Conversion").  Builds the
 * chunk table, the shard->canonical gather segments (affine maps and the
 * fused-QKV de-interleave), the canonical->receiver scatter segments
 * (including row-group remaps), the windows and the plan hash, and uploads
 * them to the current CUDA device.  *out is owned by the caller and freed
 * with dcr_plan_destroy.  Errors: DCR_ERR_INVALID (bad descriptor: unknown
 * dtype/split, tp > 16, shapes not divisible by tp or by the row group,
 * odd e2m1 shard columns), DCR_ERR_NOMEM, DCR_ERR_CUDA. */
int dcr_plan_build(const dcr_tensor_desc* tensors, size_t n, const dcr_plan_opts* opts,
                   dcr_plan** out);
int dcr_plan_info_get(const dcr_plan* plan, dcr_plan_info* out);
int dcr_window_info_get(const dcr_plan* plan, uint32_t window, dcr_window_info* out);
void dcr_plan_destroy(dcr_plan* plan);

/* Receiver state (paper summary, "Recoverable in-place apply"; popular
 * write-up on dedup by unique IDs and joint commit): the committed version
 * and, per chunk, the version it was last claimed for with NOT_STARTED /
 * CLAIMED / DONE, kept in device memory.  A frame's dedup ID is
 * (target_version, chunk_id).  Freed with dcr_recv_state_destroy. */
int dcr_recv_state_create(const dcr_plan* plan, uint64_t version, dcr_recv_state** out);
void dcr_recv_state_destroy(dcr_recv_state* state);
int dcr_recv_state_version(const dcr_recv_state* state, uint64_t* out);

/* Encode one window (blog, "Delta update algebra"; paper summary, "Hybrid
 * encoding and compression"; paper abstract).  old_shards[r] / new_shards[r]
 * are the trainer arenas of shard r (device, read only).  For each chunk:
 * gather old and new through the plan, mask = old XOR new, count changed
 * elements, then emit an XOR_LZ4 frame (XOR_SNAPPY with the plan's Snappy
 * codec; XOR_RAW if the block is not smaller) for
 * affine tensors, or OVERWRITE records (OVERWRITE_DENSE if not smaller) for
 * residual tensors and in DCR_MODE_OVERWRITE_ONLY.  The stream is written to
 * `payload` (device, payload_cap bytes); *payload_size gets its size.
 * changed_per_tensor (host, n_tensors entries, nullable) receives the changed
 * element counts of this window.  Errors: DCR_ERR_INVALID, DCR_ERR_CAPACITY
 * (*payload_size = bytes required; the window's payload_bound always fits),
 * DCR_ERR_CUDA, DCR_ERR_TIMEOUT. */
int dcr_encode(const dcr_plan* plan, uint32_t mode, uint32_t window,
               const void* const* old_shards, const void* const* new_shards,
               uint64_t base_version, uint64_t target_version,
               void* payload, size_t payload_cap, size_t* payload_size,
               uint64_t* changed_per_tensor, void* stream);

/* Apply one window's stream in place (paper summary, "Recoverable in-place
 * apply"; popular write-up on in-place apply without a backup and on dedup).
 * `payload` (device, `size` bytes) is checked against the plan hash and the
 * state's version before any byte of `target` (device receiver arena) is
 * touched.  XOR frames claim their chunk and are skipped if it was already
 * claimed for this target version; overwrite frames always apply.  The
 * version advances to target_version once every window of it has all its
 * framed chunks DONE.  fault is test only (nullable); result is nullable.
 * Errors: DCR_ERR_INVALID (plan hash, window, argument), DCR_ERR_VERSION,
 * DCR_ERR_CORRUPT (malformed frames; the others are still applied; also a
 * stream that repeats overwrite frames more often than the window has
 * chunks, when the plan routes frames through its frame lists),
 * DCR_ERR_ABORTED, DCR_ERR_INCOMPLETE (claimed chunks left unfinished by an
 * earlier abort: run dcr_apply_retry), DCR_ERR_CUDA. */
int dcr_apply(const dcr_plan* plan, dcr_recv_state* state, const void* payload, size_t size,
              void* target, const dcr_fault* fault, dcr_apply_result* result, void* stream);

/* Overwrite-only retry (popular write-up: after a failure the change set is
 * re-sent as overwrites, which are idempotent; paper abstract: retries
 * overwrite partial writes).  Same as dcr_apply but accepts only streams
 * encoded with DCR_MODE_OVERWRITE_ONLY; returns DCR_ERR_INVALID otherwise,
 * before touching `target`. */
int dcr_apply_retry(const dcr_plan* plan, dcr_recv_state* state, const void* payload, size_t size,
                    void* target, dcr_apply_result* result, void* stream);

/* Overwrite-only retry stream built from the window's XOR stream (paper
 * summary, "Recoverable in-place apply": after a failure the change set is
 * sent again as idempotent overwrites; popular write-up, in-place apply
 * without a backup copy: the sender need not read old again).  xor_payload
 * (device, xor_size bytes) is a stream dcr_encode wrote for one window of
 * this plan; for every frame the mask is decoded, the changed units read off
 * it (16-bit words of bf16 tensors, bytes otherwise) and their values
 * gathered from new_shards (device, the trainer arenas of the new version);
 * frames that already are overwrite records are copied.  The stream written
 * to `payload` (device, payload_cap bytes; *payload_size its size) carries
 * the XOR stream's window and versions and equals, byte for byte, what
 * dcr_encode writes in DCR_MODE_OVERWRITE_ONLY for the same old and new,
 * without reading old: it reads the XOR stream and the changed units of
 * new.  Errors: DCR_ERR_INVALID (plan, window or arena mismatch),
 * DCR_ERR_CORRUPT (malformed or lying frames, a chunk framed twice),
 * DCR_ERR_CAPACITY (*payload_size = bytes required), DCR_ERR_CUDA. */
int dcr_encode_retry(const dcr_plan* plan, const void* xor_payload, size_t xor_size,
                     const void* const* new_shards, void* payload, size_t payload_cap, size_t* payload_size,
                     void* stream);

/* dcr_apply without allocation.  No counterpart in the method's pages: it is
 * a deployment variant for receivers that cannot allocate device memory when
 * a refit arrives (an inference engine that reserved nearly all free HBM for
 * its KV cache at start-up).  Same arguments, decode, dedup, commit rule and
 * errors as dcr_apply with fault == NULL, but the call's scratch (its
 * counters and the list of deferred frames) is a static device array of the
 * library (768 KiB + 268 B per device) instead of the receiver state's
 * buffers, and the status is read back into a stack buffer: the call
 * neither allocates nor frees device or pinned memory.
 *   - Limit: windows of at most 65536 chunks (4 GiB of canonical bytes);
 *     plans with larger windows get DCR_ERR_CAPACITY before anything runs.
 *   - The counters are cleared by a memset on `stream` at the start of each
 *     call; nothing has to be zeroed by the caller.
 *   - dcr_recv_state_create looks up the array's device address on the
 *     current device (loading the library's apply code there if it is not
 *     loaded yet, which may allocate), and dcr_plan_build loads the apply
 *     kernels: a dcr_apply_noalloc call after those loads no code and
 *     allocates nothing.  The address is kept with the CUDA context it was
 *     found in; under a new context (after cudaDeviceReset, or a released
 *     and re-created primary context) the next call looks it up again, which
 *     may load code then: create the plan and receiver state again after a
 *     reset.  Do that set-up before any stream capture.
 *   - The static scratch is shared by every call on a device, whatever the
 *     plan or receiver state: calls on one device must not overlap in time
 *     (concurrent calls race on the counters). */
int dcr_apply_noalloc(const dcr_plan* plan, dcr_recv_state* state, const void* payload, size_t size,
                      void* target, dcr_apply_result* result, void* stream);

/* Pipelined refit of every window through host memory (paper summary,
 * "Pipelined transfer": a window's stream is built while the previous one
 * is sent; popular write-up, the transfer step).  Same frames, dedup, commit
 * rule and errors as calling, window by window in order, dcr_encode, a copy
 * of the stream from device to pinned host memory and back, and dcr_apply
 * (dcr_apply_retry for DCR_MODE_OVERWRITE_ONLY); with two buffers of each
 * kind, window k's copies run on a second stream while window k+1 is encoded
 * and window k-1 applied on `stream`.  device_buf (device, 256-byte aligned)
 * and host_buf (pinned host memory from cudaMallocHost or cudaHostAlloc,
 * 256-byte aligned) are caller-owned scratch of at least the sizes
 * dcr_pipeline_sizes gives; the call returns after all its work has finished.
 * changed_per_tensor (host, n_tensors entries, nullable) gets the counts of
 * all windows; stats (nullable) the totals.  On an error the work already in
 * flight finishes first, and the receiver state records only windows whose
 * apply status was checked.  The plan keeps the call's copy stream and
 * events (created on first use): calls on one plan must not overlap, as for
 * dcr_encode.  Kernel timing (dcr_plan_last_profile) covers dcr_encode /
 * dcr_apply calls only.  Errors: DCR_ERR_INVALID (arguments,
 * buffers too small, unaligned or not pinned), the errors of dcr_encode and
 * dcr_apply, DCR_ERR_CUDA. */
typedef struct {
    uint64_t windows;             /* windows applied and checked */
    uint64_t payload_bytes;       /* stream bytes of all windows (each crossed host memory twice) */
    uint64_t max_window_payload;
    uint32_t committed;           /* 1 if target_version was committed */
    uint32_t reserved;
} dcr_pipeline_stats;
int dcr_pipeline_sizes(const dcr_plan* plan, size_t* device_bytes, size_t* host_bytes);
int dcr_refit_pipelined(const dcr_plan* plan, dcr_recv_state* state, uint32_t mode,
                        const void* const* old_shards, const void* const* new_shards,
                        uint64_t base_version, uint64_t target_version, void* target,
                        void* device_buf, size_t device_bytes, void* host_buf, size_t host_bytes,
                        uint64_t* changed_per_tensor, dcr_pipeline_stats* stats, void* stream);

/* Ownership-sharded encode (blog, "A strong baseline with the
 * Blackwell-native DE": weight ownership is remapped so that the trainer
 * ranks together cover the whole checkpoint exactly once, every rank
 * compresses the part it owns on its own GPU, and only the rank-local
 * compressed payloads are gathered).  A window's chunks are split into
 * n_parts contiguous ranges: part q holds the chunks whose first canonical
 * byte falls in [q, q + 1) * B / n_parts of the window's B bytes, so the
 * parts cover the window exactly once, in chunk order (a part may be empty).
 * The stream the parts make is the one dcr_encode writes for the window,
 * byte for byte:
 *   header (64 B) | frames of part 0 | ... | frames of part n-1 |
 *   index entries of part 0 | ... | index entries of part n-1.
 * Per rank: dcr_encode_part (sizes), an exchange of every part's
 * dcr_part_size (a gather of 16 bytes per rank), dcr_stream_layout (the
 * offsets), dcr_encode_part_write (this part's frames and index entries at
 * those offsets, into a buffer that is then gathered into the stream, or
 * into the stream itself), and dcr_stream_header by the rank that assembles
 * the stream.  No kernel reads another GPU's memory; the exchange is the
 * caller's collective.  At most DCR_MAX_PARTS parts. */
#define DCR_MAX_PARTS 65536u
typedef struct {
    uint64_t chunk_begin, chunk_count;  /* global chunk ids of the part */
    uint64_t canonical_bytes;           /* weight bytes the part encodes */
    uint32_t shard_mask;                /* bit r set: the part reads trainer shard r */
    uint32_t reserved;
} dcr_part_info;
typedef struct {
    uint64_t frame_bytes;   /* bytes of the part's frames (a multiple of 16) */
    uint64_t n_frames;      /* its frames, i.e. its index entries */
} dcr_part_size;

/* Host only (no CUDA call): the chunk range of part `part` of `n_parts` of
 * window `window`, its bytes and the trainer shards it reads.
 * Errors: DCR_ERR_INVALID. */
int dcr_part_info_get(const dcr_plan* plan, uint32_t window, uint32_t part, uint32_t n_parts,
                      dcr_part_info* out);

/* Sizing pass of one part: the same gather, XOR, counts and encode as
 * dcr_encode, over the part's chunks only, into the plan's scratch.
 * old_shards / new_shards as in dcr_encode; only the shards in the part's
 * shard_mask are read (the others may be NULL).  *size gets the part's
 * frame bytes and frame count, changed_per_tensor (host, nullable) its
 * changed counts.  The plan remembers the part (and the shard pointers)
 * until the next encode on it: keep the arenas unchanged until
 * dcr_encode_part_write.  Errors as dcr_encode (no DCR_ERR_CAPACITY). */
int dcr_encode_part(const dcr_plan* plan, uint32_t mode, uint32_t window, uint32_t part, uint32_t n_parts,
                    const void* const* old_shards, const void* const* new_shards, dcr_part_size* size,
                    uint64_t* changed_per_tensor, void* stream);

/* Write pass of the part sized last on this plan: its frames to `frames`
 * (device, 16-byte aligned, frames_cap bytes; the frame at offset o of the
 * part lands at frames + o) and its n_frames index entries, the stream
 * offsets frame_offset + o, to `index` (device, 8-byte aligned).
 * frame_offset is where `frames` sits in the stream (dcr_stream_layout's
 * frame_offsets[part]); `frames` may point there in the stream itself, or
 * into a staging buffer that the caller gathers into it.  May be called
 * again for the same part.  Errors: DCR_ERR_INVALID (no part sized,
 * alignment), DCR_ERR_CAPACITY (frames_cap < frame_bytes), DCR_ERR_CORRUPT,
 * DCR_ERR_CUDA. */
int dcr_encode_part_write(const dcr_plan* plan, uint64_t frame_offset, void* frames, size_t frames_cap,
                          void* index, void* stream);

/* Host only: where each part's frames and index entries go in the window's
 * stream (byte offsets from the stream start), from every part's size in
 * part order, and the stream's total size.  Errors: DCR_ERR_INVALID. */
int dcr_stream_layout(uint32_t n_parts, const dcr_part_size* sizes, uint64_t* frame_offsets,
                      uint64_t* index_offsets, uint64_t* total);

/* Host only: the 64-byte stream header of window `window` (host memory) for
 * a stream of n_frames frames taking frame_bytes bytes, the sums over all
 * parts.  Errors: DCR_ERR_INVALID. */
int dcr_stream_header(const dcr_plan* plan, uint32_t mode, uint32_t window, uint64_t base_version,
                      uint64_t target_version, uint64_t n_frames, uint64_t frame_bytes, void* header);

/* Kernel timing (tracing aid).  When on, the library records CUDA events on
 * the caller's stream around each of its kernels; dcr_plan_last_profile
 * returns the durations in milliseconds of the kernels of the latest
 * dcr_encode (encode_ms, finalize_ms) and of the latest dcr_apply /
 * dcr_apply_retry (apply_ms, defer_ms, pending_ms), valid = 1 if measured;
 * the durations are read from the events when it is called, so one call
 * after an encode and its apply returns both.  The record is per plan; off
 * by default. */
typedef struct {
    float encode_ms;    /* gather + XOR + count + encode + frame write (main kernel) */
    float finalize_ms;  /* spilled (dense) chunk bodies, frame index, stream header */
    float apply_ms;     /* first phase: routing, warp- / CTA- / thread-per-frame walks */
    float defer_ms;     /* deferred frames: general blocks, bitmap walk (0 if none) */
    float pending_ms;   /* commit check */
    uint32_t encode_valid, apply_valid;
    uint32_t encode_kernels, apply_kernels;   /* kernels those calls launched */
} dcr_profile;
int dcr_plan_set_profiling(dcr_plan* plan, int on);
int dcr_plan_last_profile(const dcr_plan* plan, dcr_profile* out);

/* Dense refit: copy every canonical byte from the trainer arenas into the
 * receiver arena (the full-checkpoint transfer the delta refit replaces;
 * also how a receiver is first filled).  No status read, no sync. */
int dcr_dense_refit(const dcr_plan* plan, const void* const* shards, void* target, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DCR_H */
