// Internal definitions shared by the DCR library's host plan builder and its
// CUDA kernels (not part of the public C ABI in include/dcr.h).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <string>
#include <vector>

#include "../../include/dcr.h"

namespace dcr {

constexpr uint32_t kChunk = DCR_CHUNK_BYTES;
constexpr uint32_t kStreamHdr = DCR_STREAM_HEADER_BYTES;
constexpr uint32_t kFrameHdr = DCR_FRAME_HEADER_BYTES;
constexpr uint32_t kStreamMagic = 0x53524344u;  // "DCRS"
constexpr uint32_t kFrameMagic = 0x46524344u;   // "DCRF"
constexpr uint32_t kFormat = 1;
constexpr uint32_t kStreamOverwriteOnly = 1;
constexpr uint32_t kFrameZsrc = 1;  // every LZ4 match copies zero bytes
enum FrameKind : uint32_t { kXorLz4 = 1, kXorRaw = 2, kOverwrite = 3, kOverwriteDense = 4, kXorSnappy = 5 };

// One contiguous piece of a chunk: canonical bytes [off, off + len) of the
// chunk map to `addr`.  Sender pieces: addr = shard << 56 | byte offset in
// that shard's arena.  Receiver pieces: byte offset in the receiver arena.
struct Seg {
    uint32_t off;
    uint32_t len;
    uint64_t addr;
};
constexpr int kShardShift = 56;
constexpr uint64_t kAddrMask = (1ull << kShardShift) - 1;

enum ChunkFlags : uint32_t {
    kSrcVec = 1,  // every sender piece 16-byte aligned (offset, length, address)
    kDstVec = 2,  // every receiver piece 16-byte aligned
};

struct ChunkDesc {
    uint32_t src_begin, src_count;
    uint32_t dst_begin, dst_count;
    uint32_t raw_len;
    uint32_t tensor;     // index of the tensor descriptor (changed counts)
    uint32_t bits;       // 16, 8 or 4
    uint32_t flags;      // ChunkFlags | residual << 8
};
constexpr uint32_t kResidualFlag = 1u << 8;

// Frame offset record of one chunk of the window being encoded (written by
// the frame-size scan): bits 40-63 frames before it, bits 0-39 frame bytes
// before it.  Both fields stay in range for a window of at most 256 GiB
// (2^22 chunks, < 2^40 frame bytes).
constexpr int kLbFrameShift = 40;
constexpr uint64_t kLbByteMask = (1ull << kLbFrameShift) - 1;
constexpr uint64_t kMaxWindowBytes = 256ull << 30;

// Device scratch of one encode call (reset by a memset per call).
struct EncScratch {
    uint32_t ticket;
    int32_t err;
    uint64_t total;     // stream bytes
    uint64_t n_frames;
    uint64_t changed;   // changed elements in the window
    uint32_t n_spill;        // chunks whose frame body did not fit its slot
    uint32_t spill_ticket;   // restream pass: next spill record
    uint32_t n_deep;         // spill records left to the spill kernel
    uint32_t scan_ticket;    // scan_kernel: next tile
    uint64_t heap_top;       // bytes reserved in the overflow heap
};

// scan_kernel tiles: 8192 chunks each.  Per tile, a status word: bits 62-63
// 1 = the tile's own sum published, 2 = the inclusive prefix through the
// tile published; bits 0-61 the value (frames << 40 | frame bytes).
constexpr uint32_t kScanTile = 8192;
constexpr uint64_t kTileAgg = 1ull << 62;
constexpr uint64_t kTileInc = 2ull << 62;
constexpr uint64_t kTileValMask = (1ull << 62) - 1;

// The encoder writes each chunk's frame into a slot of its own in device
// scratch (kEncSlot bytes per chunk of the window); a compaction pass copies
// the slots into the stream once the frame offsets are known.
constexpr uint32_t kEncSlot = 6144;
constexpr uint32_t kSpilled = 1u << 31;   // frame-size flag: body not in the slot (write pass re-derives it)
constexpr uint32_t kHeap = 1u << 30;      // frame-size flag: the frame goes on past the slot, in the heap
constexpr uint32_t kFrameSizeMask = kHeap - 1;
// A warp's overflow buffer: the part of an XOR block past its slot, moved
// to the heap at the chunk's end.
constexpr uint32_t kOvfBytes = 65536;

// A chunk whose frame is sized but whose body did not fit its slot: a
// restream pass re-derives it and writes the frame into the stream (the
// spill kernel takes raw and dense frames and LZ4 chunks with very long
// literal runs).
struct SpillRec {
    uint32_t k;          // window-relative chunk
    uint32_t kind;       // FrameKind
    uint32_t body_len;
    uint32_t n_units;    // overwrite records: unit count
    uint32_t changed;    // changed stored values (frame header)
    uint32_t pad[3];
};

// Device scratch of one apply call (reset by a memset per call).
struct ApplyScratch {
    int32_t err;
    uint32_t hdr_ok;
    uint32_t frame_ticket;
    uint32_t n_defer;
    uint32_t defer_ticket;
    uint32_t aborted;
    uint32_t window;
    uint32_t n_big;         // large ZSRC frames, listed from the end of the deferred list
    unsigned long long applied;
    unsigned long long skipped;
    unsigned long long pending;
    uint64_t target_version;
    uint64_t n_frames;
    uint32_t big_ticket;
    uint32_t n_lane;        // ZSRC frames listed for lane_kernel
    uint32_t n_warp;        // frames route_kernel lists for apply_kernel
};

// Chunk state of a receiver: (target_version << 2) | state.
enum ChunkState : uint64_t { kNotStarted = 0, kClaimed = 1, kDone = 2 };

struct Part {
    uint32_t desc, sub, residual, bits;
    uint64_t rows, cols, bytes, recv_off;
    uint64_t chunk0, nchunks;
};

struct KernelConfig {
    int num_sms = 0;
    int enc_blocks_per_sm = 0;
    int enc_deep_blocks_per_sm = 0;
    int retry_blocks_per_sm = 0;
    int enc_warps_per_block = 0;        // one chunk per warp: the wide and deep variants
    int enc_deep_warps_per_block = 0;
    int restream_blocks_per_sm = 0;
    int spill_blocks_per_sm = 0;
    int apply_blocks_per_sm = 0;
    int apply_cta_blocks_per_sm = 0;
    int defer_blocks_per_sm = 0;
    int big_blocks_per_sm = 0;
    int split_blocks_per_sm = 0;       // big_kernel with the split walk (Snappy plans)
    int lane_blocks_per_sm = 0;
};

// host entry points of the kernel translation units
int encode_launch(const struct ::dcr_plan* plan, uint32_t mode, uint32_t window,
                  const void* const* olds, const void* const* news, uint64_t base_version,
                  uint64_t target_version, void* payload, size_t cap, cudaStream_t s);
// the two passes of one encode over a chunk range, for ownership-sharded
// encodes: sizing (frames into slots, sizes scanned) and writing (frames to
// `frames`, index entries frame_base + offset to `index`)
int encode_size_launch(const struct ::dcr_plan* plan, uint32_t mode, uint64_t chunk_begin, uint64_t chunk_count,
                       const void* const* olds, const void* const* news, cudaStream_t s);
int encode_write_launch(const struct ::dcr_plan* plan, uint32_t mode, uint64_t chunk_begin, uint64_t chunk_count,
                        const void* const* olds, const void* const* news, uint8_t* frames, uint64_t frame_base,
                        uint64_t* index, cudaStream_t s);
// dcr_encode_retry: the overwrite-only stream of a window from its XOR
// stream (in, index at in_idx, in_frames frames) and new
int retry_launch(const struct ::dcr_plan* plan, const void* in, uint64_t in_idx, uint64_t in_frames,
                 uint32_t window, uint64_t base_v, uint64_t target_v, const void* const* news, void* payload,
                 size_t cap, cudaStream_t s);
int encode_kernel_config(KernelConfig* kc);
int apply_kernel_config(KernelConfig* kc);
int apply_launch(const struct ::dcr_plan* plan, struct ::dcr_recv_state* st, const void* payload,
                 size_t size, void* target, uint64_t abort_at, uint32_t split, int retry_only,
                 cudaStream_t s);
// one part of an apply: kApplyFirst = the first kernel and the commit check;
// kApplyDeferred = the deferred-frame kernels and the commit check again;
// kApplyAll = all of them (what apply_launch launches)
enum { kApplyAll = 0, kApplyFirst = 1, kApplyDeferred = 2 };
// kernels one call launches: dcr_encode (encode, scan, copy, restream,
// spill), dcr_encode_retry (retry walk, retry, scan, copy, retry spill,
// retry write, retry values); dcr_apply counts its own
// (dcr_plan::apply_kernels)
constexpr uint32_t kEncodeKernels = 5, kRetryKernels = 7;
int apply_launch_part(const struct ::dcr_plan* plan, struct ::dcr_recv_state* st, const void* payload,
                      size_t size, void* target, uint64_t abort_at, uint32_t split, int retry_only, int part,
                      cudaStream_t s);
int dense_launch(const struct ::dcr_plan* plan, const void* const* shards, void* target,
                 cudaStream_t s);

// status of one encode / apply from the host mirror of its device scratch
int encode_result(const struct ::dcr_plan* plan, const void* head, size_t cap, size_t* payload_size,
                  uint64_t* changed, bool accumulate);
int apply_result(struct ::dcr_recv_state* st, const ApplyScratch& a, dcr_apply_result* result);

void pipe_release(const struct ::dcr_plan* plan);
// looks up dcr_apply_noalloc's static scratch for the current device and
// context (loading its module), so that the call itself allocates nothing
int noalloc_prepare();

int set_error(int code, const char* fmt, ...);
int cuda_error(cudaError_t e, const char* what);

}  // namespace dcr

struct dcr_plan {
    std::vector<dcr_tensor_desc> descs;
    std::vector<std::string> names;
    std::vector<dcr::Part> parts;
    std::vector<dcr::ChunkDesc> chunks;
    std::vector<uint64_t> win_start;  // n_windows + 1 chunk ids
    std::vector<uint64_t> chunk_start;   // canonical byte offset of each chunk in the model (+ total)
    std::vector<uint32_t> chunk_shards;  // per chunk: bit r set iff it reads trainer shard r
    bool host_only = false;              // built with DCR_PLAN_HOST_ONLY: no device state
    bool stall_scan = false;             // DCR_PLAN_TEST_STALL_SCAN: scan tile 0 never publishes
    uint64_t window_bytes = 0;
    uint32_t encoder = DCR_ENCODER_AUTO;
    uint32_t codec = DCR_CODEC_LZ4;
    uint32_t apply = DCR_APPLY_AUTO;
    int small_window_chunks = 0;         // AUTO takes the CTA-per-chunk kernels up to this window size
    uint64_t n_chunks = 0;
    uint64_t canonical_bytes = 0;
    uint64_t hash = 0;
    uint64_t recv_bytes = 0;
    uint64_t shard_bytes[DCR_MAX_TP] = {};
    uint32_t tp = 1;
    uint64_t max_window_chunks = 0;
    int device = 0;
    dcr::KernelConfig kc;
    // device tables
    dcr::ChunkDesc* d_chunks = nullptr;
    dcr::Seg* d_src = nullptr;
    dcr::Seg* d_dst = nullptr;
    uint64_t* d_win = nullptr;         // n_windows + 1 chunk ids
    uint64_t n_src = 0, n_dst = 0;
    // encode scratch: [EncScratch][u64 counts[n_tensors]] then lb[], fsize[]
    void* d_enc = nullptr;
    size_t enc_head_bytes = 0;
    uint64_t* d_lb = nullptr;
    uint32_t* d_fsize = nullptr;
    dcr::SpillRec* d_spill = nullptr;  // max_window_chunks
    uint32_t* d_deep = nullptr;        // max_window_chunks spill record ids
    uint64_t* d_tiles = nullptr;       // scan_kernel tile status words
    uint8_t* d_ovf = nullptr;          // per-warp overflow buffers of the one-warp encoders
    uint8_t* d_heap = nullptr;         // rests of bodies past their slots
    uint64_t heap_bytes = 0;
    uint64_t* d_heapoff = nullptr;     // max_window_chunks heap offsets
    mutable bool overflow_seen = false;   // an encode on this plan had a body outgrow its slot
    uint32_t max_tiles = 0;
    uint8_t* d_slots = nullptr;        // max_window_chunks * kEncSlot frame slots
    void* h_enc = nullptr;  // pinned mirror of the scratch head
    // kernel timing (dcr_plan_set_profiling)
    bool profiling = false;
    cudaEvent_t ev[8] = {};
    mutable dcr_profile prof = {};
    mutable bool prof_encode_due = false, prof_apply_due = false;   // events recorded, durations not read
    mutable bool prof_deferred = false;   // the deferred-frame kernels ran after a status read (from ev[7])
    mutable uint32_t apply_kernels = 0;   // kernels the latest apply launched
    // ownership-sharded encode: the part sized by the last dcr_encode_part
    struct {
        bool valid = false;
        uint32_t mode = 0, window = 0;
        uint64_t chunk_begin = 0, chunk_count = 0, frame_bytes = 0, n_frames = 0;
        const void* olds[DCR_MAX_TP] = {};
        const void* news[DCR_MAX_TP] = {};
    } mutable part;
    // dcr_refit_pipelined: its copy stream and events (created on first use)
    mutable cudaStream_t pipe_copy = nullptr;
    mutable cudaEvent_t pipe_ev[8] = {};
};

struct dcr_recv_state {
    const dcr_plan* plan = nullptr;
    uint64_t version = 0;
    uint64_t pending = ~0ull;
    std::vector<uint8_t> win_done;
    uint64_t* d_chunk_state = nullptr;  // n_chunks
    dcr::ApplyScratch* d_scratch = nullptr;
    uint32_t* d_defer = nullptr;        // 3 x (max_window_chunks + 1): deferred frames, lane and warp lists
    dcr::ApplyScratch* h_scratch = nullptr;  // pinned
};
