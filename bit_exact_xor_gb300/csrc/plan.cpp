// Host side of the DCR library: plan build (chunk table, gather/scatter
// segments, windows, plan hash), receiver state, error reporting, and the C
// ABI wrappers around the kernel launchers.
//
// The plan is the host-prepared apply metadata of "GPU-accelerated weight
// teleportation" ("A strong baseline with the Blackwell-native DE": tiling
// and address mapping prepared on the CPU, read by the kernel; "Working with
// low-precision RL": the mask is remapped like the weights' physical layout)
// together with the fixed shard -> canonical maps of the NeMo-DCR paper
// summary ("Direct Projection", "Residual Conversion").
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>

#include "dcr_internal.h"

namespace dcr {

static thread_local char g_err[512] = "no error";

int set_error(int code, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int cuda_error(cudaError_t e, const char* what)
{
    return set_error(DCR_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

namespace {

bool desc_ok(const dcr_tensor_desc& d, const char** why)
{
    *why = nullptr;
    if (d.elem_bits != 4 && d.elem_bits != 8 && d.elem_bits != 16) *why = "elem_bits must be 4, 8 or 16";
    else if (d.tp < 1 || d.tp > DCR_MAX_TP) *why = "tp must be 1..16";
    else if (d.rows == 0 || d.cols == 0) *why = "empty tensor";
    else if (d.elem_bits == 4 && d.cols % 2) *why = "e2m1 tensors need an even column count";
    else if (d.split == DCR_SPLIT_ROWS && d.rows % d.tp) *why = "rows not divisible by tp";
    else if (d.split == DCR_SPLIT_COLS && d.cols % d.tp) *why = "cols not divisible by tp";
    else if (d.split == DCR_SPLIT_COLS && d.elem_bits == 4 && (d.cols / d.tp) % 2)
        *why = "e2m1 shard columns must be even";
    else if (d.split == DCR_RESIDUAL_QKV_INTERLEAVED) {
        if (!d.q_heads || !d.kv_heads || !d.head_dim) *why = "qkv needs head counts";
        else if (d.q_heads % d.kv_heads || d.kv_heads % d.tp) *why = "qkv head counts not divisible";
        else if (d.rows != (uint64_t)(d.q_heads + 2ull * d.kv_heads) * d.head_dim)
            *why = "qkv rows != (q + 2 kv) * head_dim";
        else if (d.recv_layout != DCR_LAYOUT_CANONICAL) *why = "qkv receiver layout must be canonical";
    } else if (d.split > DCR_SPLIT_COLS) *why = "unknown split";
    if (!*why) {
        if (d.recv_layout == DCR_LAYOUT_ROWGROUP_INTERLEAVE) {
            if (!d.recv_group || d.rows % d.recv_group || d.recv_slot > 1) *why = "bad row-group layout";
        } else if (d.recv_layout != DCR_LAYOUT_CANONICAL) {
            *why = "unknown receiver layout";
        }
    }
    return *why == nullptr;
}

struct Hash {
    uint64_t h = 0xCBF29CE484222325ull;
    void bytes(const void* p, size_t n)
    {
        const uint8_t* b = static_cast<const uint8_t*>(p);
        for (size_t i = 0; i < n; ++i) { h ^= b[i]; h *= 0x100000001B3ull; }
    }
    void u32(uint32_t v)
    {
        uint8_t b[4] = {uint8_t(v), uint8_t(v >> 8), uint8_t(v >> 16), uint8_t(v >> 24)};
        bytes(b, 4);
    }
    void u64(uint64_t v) { u32(uint32_t(v)); u32(uint32_t(v >> 32)); }
};

// Sender map: canonical byte x of part p -> (shard, arena byte), and the end
// of the canonical run that stays contiguous in that shard.
struct Where { uint32_t shard; uint64_t addr; uint64_t run_end; };

Where src_where(const dcr_tensor_desc& d, const Part& p, uint64_t x)
{
    const uint64_t rb = p.cols * p.bits / 8;
    Where w{0, 0, p.bytes};
    uint64_t local = x;
    switch (d.split) {
    case DCR_REPLICATED:
        break;
    case DCR_SPLIT_ROWS: {
        uint64_t sb = (d.rows / d.tp) * rb;
        w.shard = uint32_t(x / sb);
        local = x % sb;
        w.run_end = (x / sb + 1) * sb;
        break;
    }
    case DCR_SPLIT_COLS: {
        uint64_t lb = rb / d.tp, q = x / lb;
        w.shard = uint32_t(q % d.tp);
        local = (q / d.tp) * lb + x % lb;
        w.run_end = (q + 1) * lb;
        break;
    }
    default: {  // fused QKV: shard r holds kv groups [r*G/tp, (r+1)*G/tp)
        uint64_t D = d.head_dim, G = d.kv_heads, qpg = d.q_heads / G, gpl = G / d.tp;
        uint64_t row = x / rb, g, rig, blk_rows;
        if (p.sub == 0) {
            g = row / (qpg * D);
            rig = row % (qpg * D);
            blk_rows = (g + 1) * qpg * D;
        } else {
            g = row / D;
            rig = (qpg + p.sub - 1) * D + row % D;
            blk_rows = (g + 1) * D;
        }
        w.shard = uint32_t(g / gpl);
        local = ((g % gpl) * (qpg + 2) * D + rig) * rb + x % rb;
        w.run_end = blk_rows * rb;
        break;
    }
    }
    w.addr = d.shard_offset[w.shard] + local;
    return w;
}

// Receiver map: canonical byte x of part p -> receiver arena byte.
Where dst_where(const dcr_tensor_desc& d, const Part& p, uint64_t x)
{
    Where w{0, p.recv_off + x, p.bytes};
    if (d.recv_layout == DCR_LAYOUT_ROWGROUP_INTERLEAVE) {
        const uint64_t rb = p.cols * p.bits / 8, g = d.recv_group;
        uint64_t row = x / rb, grp = row / g;
        uint64_t prow = grp * 2 * g + d.recv_slot * g + row % g;
        w.addr = p.recv_off + prow * rb + x % rb;
        w.run_end = (grp + 1) * g * rb;
    }
    return w;
}

template <class F>
void cut(const Part& p, uint64_t off, uint32_t len, F where, std::vector<Seg>& out, bool* vec)
{
    size_t first = out.size();
    uint64_t x = off, end = off + len;
    while (x < end) {
        Where w = where(x);
        uint64_t e = w.run_end < end ? w.run_end : end;
        uint64_t a = (uint64_t(w.shard) << kShardShift) | w.addr;
        if (out.size() > first) {
            Seg& b = out.back();
            if (b.addr + b.len == a && ((b.addr >> kShardShift) == w.shard)) {
                b.len += uint32_t(e - x);
                x = e;
                continue;
            }
        }
        out.push_back(Seg{uint32_t(x - off), uint32_t(e - x), a});
        x = e;
    }
    bool v = len % 16 == 0;
    for (size_t i = first; i < out.size(); ++i)
        v = v && out[i].off % 16 == 0 && out[i].len % 16 == 0 && (out[i].addr & kAddrMask) % 16 == 0;
    *vec = v;
}

template <class T>
int upload(T** dptr, const std::vector<T>& v)
{
    size_t n = v.empty() ? 1 : v.size();
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(dptr), n * sizeof(T));
    if (e != cudaSuccess) return cuda_error(e, "cudaMalloc(plan table)");
    if (!v.empty()) {
        e = cudaMemcpy(*dptr, v.data(), v.size() * sizeof(T), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_error(e, "cudaMemcpy(plan table)");
    }
    return DCR_OK;
}

void plan_free_device(dcr_plan* p)
{
    for (cudaEvent_t& e : p->ev) {
        if (e) cudaEventDestroy(e);
        e = nullptr;
    }
    pipe_release(p);
    cudaFree(p->d_chunks);
    cudaFree(p->d_src);
    cudaFree(p->d_dst);
    cudaFree(p->d_win);
    p->d_win = nullptr;
    cudaFree(p->d_enc);
    cudaFree(p->d_slots);
    cudaFree(p->d_ovf);
    cudaFree(p->d_heap);
    cudaFree(p->d_heapoff);
    p->d_ovf = p->d_heap = nullptr;
    p->d_heapoff = nullptr;
    if (p->h_enc) cudaFreeHost(p->h_enc);
    p->d_chunks = nullptr;
    p->d_src = p->d_dst = nullptr;
    p->d_enc = nullptr;
    p->d_slots = nullptr;
    p->h_enc = nullptr;
}

}  // namespace
}  // namespace dcr

using namespace dcr;

extern "C" const char* dcr_last_error(void) { return g_err; }

extern "C" int dcr_plan_build(const dcr_tensor_desc* tensors, size_t n, const dcr_plan_opts* opts,
                              dcr_plan** out)
{
    if (!out) return set_error(DCR_ERR_INVALID, "dcr_plan_build: out is NULL");
    *out = nullptr;
    if (!tensors || n == 0) return set_error(DCR_ERR_INVALID, "dcr_plan_build: no tensors");
    uint64_t W = opts && opts->window_bytes ? opts->window_bytes : (16ull << 30);
    if (W < kChunk || W > kMaxWindowBytes)
        return set_error(DCR_ERR_INVALID, "window_bytes must be in [64 KiB, 256 GiB]");
    const uint32_t encoder = opts ? opts->encoder : uint32_t(DCR_ENCODER_AUTO);
    if (encoder > DCR_ENCODER_CTA) return set_error(DCR_ERR_INVALID, "unknown encoder variant %u", encoder);
    const uint32_t codec = opts ? opts->codec : uint32_t(DCR_CODEC_LZ4);
    if (codec > DCR_CODEC_SNAPPY) return set_error(DCR_ERR_INVALID, "unknown codec %u", codec);
    const uint32_t flags = opts ? opts->flags : 0u;
    const uint32_t apply = opts ? opts->apply : uint32_t(DCR_APPLY_AUTO);
    const uint32_t overflow_kib = opts ? opts->overflow_kib : 0u;
    if (apply > DCR_APPLY_SPLIT) return set_error(DCR_ERR_INVALID, "unknown apply variant %u", apply);
    if (flags & ~uint32_t(DCR_PLAN_HOST_ONLY | DCR_PLAN_TEST_STALL_SCAN))
        return set_error(DCR_ERR_INVALID, "unknown plan flags %#x", flags);
    dcr_plan* P = new (std::nothrow) dcr_plan();
    if (!P) return set_error(DCR_ERR_NOMEM, "dcr_plan_build: out of host memory");
    P->window_bytes = W;
    P->host_only = (flags & DCR_PLAN_HOST_ONLY) != 0;
    P->stall_scan = (flags & DCR_PLAN_TEST_STALL_SCAN) != 0;
    P->encoder = encoder;
    P->codec = codec;
    P->apply = apply;
    P->tp = tensors[0].tp;
    for (size_t i = 0; i < n; ++i) {
        const char* why;
        if (!desc_ok(tensors[i], &why)) {
            delete P;
            return set_error(DCR_ERR_INVALID, "tensor %zu (%s): %s", i,
                             tensors[i].name ? tensors[i].name : "?", why);
        }
        if (tensors[i].tp > P->tp) P->tp = tensors[i].tp;
        P->descs.push_back(tensors[i]);
        P->names.emplace_back(tensors[i].name ? tensors[i].name : "");
    }
    for (size_t i = 0; i < n; ++i) P->descs[i].name = P->names[i].c_str();

    // canonical parts and chunks (64 KiB of each part's own byte space)
    uint64_t chunks = 0;
    for (size_t i = 0; i < n; ++i) {
        const dcr_tensor_desc& d = P->descs[i];
        int nsub = d.split == DCR_RESIDUAL_QKV_INTERLEAVED ? 3 : 1;
        uint64_t roff = d.recv_offset;
        for (int s = 0; s < nsub; ++s) {
            Part p{};
            p.desc = uint32_t(i);
            p.sub = uint32_t(s);
            p.bits = d.elem_bits;
            p.cols = d.cols;
            p.residual = d.split == DCR_RESIDUAL_QKV_INTERLEAVED;
            p.rows = p.residual ? uint64_t(s == 0 ? d.q_heads : d.kv_heads) * d.head_dim : d.rows;
            p.bytes = p.rows * p.cols * p.bits / 8;
            p.recv_off = roff;
            roff += p.bytes;
            p.chunk0 = chunks;
            p.nchunks = (p.bytes + kChunk - 1) / kChunk;
            chunks += p.nchunks;
            P->canonical_bytes += p.bytes;
            P->parts.push_back(p);
        }
    }
    P->n_chunks = chunks;
    if (chunks >= (1ull << 32)) {
        delete P;
        return set_error(DCR_ERR_INVALID, "too many chunks");
    }

    // windows: whole tensors in order while they fit; big tensors cut at chunks
    {
        uint64_t cur = 0;
        size_t p = 0;
        P->win_start.push_back(0);
        for (size_t i = 0; i < n; ++i) {
            size_t pe = p;
            uint64_t B = 0;
            while (pe < P->parts.size() && P->parts[pe].desc == i) B += P->parts[pe++].bytes;
            if (cur > 0 && cur + B > W) {
                P->win_start.push_back(P->parts[p].chunk0);
                cur = 0;
            }
            for (; p < pe; ++p) {
                const Part& q = P->parts[p];
                for (uint64_t c = 0; c < q.nchunks; ++c) {
                    uint64_t len = q.bytes - c * kChunk;
                    if (len > kChunk) len = kChunk;
                    if (cur > 0 && cur + len > W) {
                        P->win_start.push_back(q.chunk0 + c);
                        cur = 0;
                    }
                    cur += len;
                }
            }
        }
        P->win_start.push_back(chunks);
        for (size_t w = 0; w + 1 < P->win_start.size(); ++w) {
            uint64_t c = P->win_start[w + 1] - P->win_start[w];
            if (c > P->max_window_chunks) P->max_window_chunks = c;
        }
    }

    // plan hash over what both ends must agree on (canonical description)
    {
        Hash h;
        h.bytes("DCR1", 4);
        h.u32(kChunk);
        h.u64(W);
        h.u32(uint32_t(P->parts.size()));
        for (const Part& q : P->parts) {
            h.u32(q.bits);
            h.u64(q.rows);
            h.u64(q.cols);
            h.u32(q.residual);
            h.u32(q.desc);
        }
        P->hash = h.h;
    }

    // chunk table with sender and receiver segments
    std::vector<Seg> src, dst;
    P->chunks.resize(chunks);
    P->chunk_start.resize(chunks + 1);
    P->chunk_shards.resize(chunks);
    for (const Part& q : P->parts) {
        const dcr_tensor_desc& d = P->descs[q.desc];
        for (uint64_t c = 0; c < q.nchunks; ++c) {
            uint64_t off = c * kChunk;
            uint32_t len = uint32_t(q.bytes - off < kChunk ? q.bytes - off : kChunk);
            ChunkDesc& cd = P->chunks[q.chunk0 + c];
            bool sv, dv;
            cd.src_begin = uint32_t(src.size());
            cut(q, off, len, [&](uint64_t x) { return src_where(d, q, x); }, src, &sv);
            cd.src_count = uint32_t(src.size() - cd.src_begin);
            cd.dst_begin = uint32_t(dst.size());
            cut(q, off, len, [&](uint64_t x) { return dst_where(d, q, x); }, dst, &dv);
            cd.dst_count = uint32_t(dst.size() - cd.dst_begin);
            cd.raw_len = len;
            cd.tensor = q.desc;
            cd.bits = q.bits;
            cd.flags = (sv ? kSrcVec : 0u) | (dv ? kDstVec : 0u) | (q.residual ? kResidualFlag : 0u);
            uint32_t mask = 0;
            for (uint32_t k = cd.src_begin; k < cd.src_begin + cd.src_count; ++k) {
                uint32_t r = uint32_t(src[k].addr >> kShardShift);
                uint64_t e = (src[k].addr & kAddrMask) + src[k].len;
                if (e > P->shard_bytes[r]) P->shard_bytes[r] = e;
                mask |= 1u << r;
            }
            P->chunk_shards[q.chunk0 + c] = mask;
            for (uint32_t k = cd.dst_begin; k < cd.dst_begin + cd.dst_count; ++k)
                if (dst[k].addr + dst[k].len > P->recv_bytes) P->recv_bytes = dst[k].addr + dst[k].len;
        }
    }
    if (src.size() >= (1ull << 32) || dst.size() >= (1ull << 32)) {
        delete P;
        return set_error(DCR_ERR_INVALID, "too many segments");
    }
    P->n_src = src.size();
    P->n_dst = dst.size();
    for (uint64_t c = 0; c < chunks; ++c) P->chunk_start[c + 1] = P->chunk_start[c] + P->chunks[c].raw_len;
    if (P->host_only) {   // layout, windows, hash and parts only: nothing on a device
        *out = P;
        return DCR_OK;
    }

    cudaError_t e = cudaGetDevice(&P->device);
    if (e != cudaSuccess) { delete P; return cuda_error(e, "cudaGetDevice"); }
    int rc;
    if ((rc = upload(&P->d_chunks, P->chunks)) || (rc = upload(&P->d_src, src)) ||
        (rc = upload(&P->d_dst, dst)) || (rc = upload(&P->d_win, P->win_start))) {
        plan_free_device(P);
        delete P;
        return rc;
    }
    // encode scratch: head = EncScratch + per-tensor counts, then frame
    // offsets, sizes, the spill list and the spill kernel's share of it
    P->enc_head_bytes = (sizeof(EncScratch) + 8 * n + 255) / 256 * 256;
    size_t lb_bytes = (P->max_window_chunks * 8 + 255) / 256 * 256;
    size_t fs_bytes = (P->max_window_chunks * 4 + 255) / 256 * 256;
    size_t sp_bytes = (P->max_window_chunks * sizeof(SpillRec) + 255) / 256 * 256;
    P->max_tiles = uint32_t((P->max_window_chunks + kScanTile - 1) / kScanTile + 1);
    size_t dp_bytes = (P->max_window_chunks * 4 + 255) / 256 * 256;
    size_t total = P->enc_head_bytes + lb_bytes + fs_bytes + sp_bytes + dp_bytes + P->max_tiles * 8ull + 256;
    if ((e = cudaMalloc(&P->d_enc, total)) != cudaSuccess ||
        (e = cudaMalloc(&P->d_slots, P->max_window_chunks * size_t(kEncSlot))) != cudaSuccess ||
        (e = cudaMallocHost(&P->h_enc, P->enc_head_bytes)) != cudaSuccess) {
        plan_free_device(P);
        delete P;
        return cuda_error(e, "allocating encode scratch");
    }
    P->d_lb = reinterpret_cast<uint64_t*>(static_cast<char*>(P->d_enc) + P->enc_head_bytes);
    P->d_fsize = reinterpret_cast<uint32_t*>(static_cast<char*>(P->d_enc) + P->enc_head_bytes + lb_bytes);
    P->d_spill = reinterpret_cast<SpillRec*>(static_cast<char*>(P->d_enc) + P->enc_head_bytes + lb_bytes +
                                             fs_bytes);
    P->d_deep = reinterpret_cast<uint32_t*>(reinterpret_cast<char*>(P->d_spill) + sp_bytes);
    P->d_tiles = reinterpret_cast<uint64_t*>(reinterpret_cast<char*>(P->d_deep) + dp_bytes);
    if ((rc = encode_kernel_config(&P->kc)) || (rc = apply_kernel_config(&P->kc))) {
        plan_free_device(P);
        delete P;
        return rc;
    }
    P->small_window_chunks = P->kc.num_sms * P->kc.enc_deep_blocks_per_sm * P->kc.enc_deep_warps_per_block;
    // overflow buffers (one per warp of the one-warp encoders) and the heap
    // that XOR bodies past their slots move to
    if (overflow_kib != DCR_NO_OVERFLOW) {
        const uint64_t warps =
            std::max<uint64_t>(uint64_t(P->kc.num_sms) * P->kc.enc_blocks_per_sm * P->kc.enc_warps_per_block,
                               uint64_t(P->kc.num_sms) * P->kc.enc_deep_blocks_per_sm * P->kc.enc_deep_warps_per_block);
        const uint64_t win = std::min<uint64_t>(W, P->canonical_bytes ? P->canonical_bytes : 1);
        P->heap_bytes = overflow_kib ? uint64_t(overflow_kib) << 10 : (win / 8 + 255) / 256 * 256;
        if ((e = cudaMalloc(&P->d_ovf, warps * kOvfBytes)) != cudaSuccess ||
            (e = cudaMalloc(&P->d_heap, P->heap_bytes ? P->heap_bytes : 256)) != cudaSuccess ||
            (e = cudaMalloc(&P->d_heapoff, (P->max_window_chunks ? P->max_window_chunks : 1) * 8)) != cudaSuccess) {
            plan_free_device(P);
            delete P;
            return cuda_error(e, "allocating the encoder's overflow heap");
        }
    }
    *out = P;
    return DCR_OK;
}

extern "C" int dcr_plan_info_get(const dcr_plan* p, dcr_plan_info* out)
{
    if (!p || !out) return set_error(DCR_ERR_INVALID, "dcr_plan_info_get: NULL argument");
    memset(out, 0, sizeof(*out));
    out->n_tensors = p->descs.size();
    out->n_parts = p->parts.size();
    out->n_chunks = p->n_chunks;
    out->n_windows = p->win_start.size() - 1;
    out->canonical_bytes = p->canonical_bytes;
    out->plan_hash = p->hash;
    out->recv_bytes = p->recv_bytes;
    for (int r = 0; r < DCR_MAX_TP; ++r) out->shard_bytes[r] = p->shard_bytes[r];
    out->tp = p->tp;
    return DCR_OK;
}

extern "C" int dcr_window_info_get(const dcr_plan* p, uint32_t w, dcr_window_info* out)
{
    if (!p || !out) return set_error(DCR_ERR_INVALID, "dcr_window_info_get: NULL argument");
    if (w + 1 >= p->win_start.size()) return set_error(DCR_ERR_INVALID, "window %u out of range", w);
    out->chunk_begin = p->win_start[w];
    out->chunk_count = p->win_start[w + 1] - p->win_start[w];
    out->canonical_bytes = 0;
    uint64_t bound = kStreamHdr;
    for (uint64_t c = out->chunk_begin; c < out->chunk_begin + out->chunk_count; ++c) {
        out->canonical_bytes += p->chunks[c].raw_len;
        bound += (kFrameHdr + p->chunks[c].raw_len + 15) / 16 * 16 + 8;
    }
    out->payload_bound = bound;
    return DCR_OK;
}

extern "C" void dcr_plan_destroy(dcr_plan* p)
{
    if (!p) return;
    if (p->host_only) {
        delete p;
        return;
    }
    int cur = -1;
    cudaGetDevice(&cur);
    if (cur != p->device) cudaSetDevice(p->device);
    plan_free_device(p);
    if (cur >= 0 && cur != p->device) cudaSetDevice(cur);
    delete p;
}

extern "C" int dcr_recv_state_create(const dcr_plan* p, uint64_t version, dcr_recv_state** out)
{
    if (!p || !out) return set_error(DCR_ERR_INVALID, "dcr_recv_state_create: NULL argument");
    *out = nullptr;
    if (p->host_only) return set_error(DCR_ERR_INVALID, "dcr_recv_state_create: host-only plan");
    dcr_recv_state* s = new (std::nothrow) dcr_recv_state();
    if (!s) return set_error(DCR_ERR_NOMEM, "dcr_recv_state_create: out of host memory");
    s->plan = p;
    s->version = version;
    s->win_done.assign(p->win_start.size() - 1, 0);
    cudaError_t e;
    if ((e = cudaMalloc(&s->d_chunk_state, (p->n_chunks ? p->n_chunks : 1) * 8)) != cudaSuccess ||
        (e = cudaMemset(s->d_chunk_state, 0, (p->n_chunks ? p->n_chunks : 1) * 8)) != cudaSuccess ||
        (e = cudaMalloc(&s->d_scratch, sizeof(ApplyScratch))) != cudaSuccess ||
        (e = cudaMalloc(&s->d_defer, 3 * (p->max_window_chunks + 1) * 4)) != cudaSuccess ||
        (e = cudaMallocHost(&s->h_scratch, sizeof(ApplyScratch))) != cudaSuccess) {
        dcr_recv_state_destroy(s);
        return cuda_error(e, "allocating receiver state");
    }
    if (int rc = noalloc_prepare()) {
        dcr_recv_state_destroy(s);
        return rc;
    }
    *out = s;
    return DCR_OK;
}

extern "C" void dcr_recv_state_destroy(dcr_recv_state* s)
{
    if (!s) return;
    cudaFree(s->d_chunk_state);
    cudaFree(s->d_scratch);
    cudaFree(s->d_defer);
    if (s->h_scratch) cudaFreeHost(s->h_scratch);
    delete s;
}

extern "C" int dcr_recv_state_version(const dcr_recv_state* s, uint64_t* out)
{
    if (!s || !out) return set_error(DCR_ERR_INVALID, "dcr_recv_state_version: NULL argument");
    *out = s->version;
    return DCR_OK;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

extern "C" int dcr_encode(const dcr_plan* p, uint32_t mode, uint32_t window,
                          const void* const* olds, const void* const* news, uint64_t base_version,
                          uint64_t target_version, void* payload, size_t cap, size_t* payload_size,
                          uint64_t* changed_per_tensor, void* stream)
{
    if (!p || !olds || !news || !payload_size)
        return set_error(DCR_ERR_INVALID, "dcr_encode: NULL argument");
    if (mode > DCR_MODE_OVERWRITE_ONLY) return set_error(DCR_ERR_INVALID, "dcr_encode: bad mode");
    if (p->host_only) return set_error(DCR_ERR_INVALID, "dcr_encode: host-only plan");
    p->part.valid = false;   // the plan's scratch now holds this encode
    if (window + 1 >= p->win_start.size())
        return set_error(DCR_ERR_INVALID, "dcr_encode: window %u out of range", window);
    if (payload && !aligned16(payload)) return set_error(DCR_ERR_INVALID, "payload not 16-byte aligned");
    for (uint32_t r = 0; r < p->tp; ++r) {
        if (p->shard_bytes[r] && (!olds[r] || !news[r]))
            return set_error(DCR_ERR_INVALID, "dcr_encode: shard %u arena is NULL", r);
        if ((olds[r] && !aligned16(olds[r])) || (news[r] && !aligned16(news[r])))
            return set_error(DCR_ERR_INVALID, "dcr_encode: shard %u arena not 16-byte aligned", r);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = encode_launch(p, mode, window, olds, news, base_version, target_version, payload,
                           payload ? cap : 0, s);
    if (rc) return rc;
    cudaError_t e = cudaMemcpyAsync(p->h_enc, p->d_enc, p->enc_head_bytes, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_error(e, "dcr_encode status read");
    if (p->profiling) {
        p->prof_encode_due = true;   // durations read from the events when asked for
        p->prof.encode_valid = 1;
        p->prof.encode_kernels = kEncodeKernels;
    }
    return encode_result(p, p->h_enc, payload ? cap : 0, payload_size, changed_per_tensor, false);
}

namespace dcr {

int encode_result(const dcr_plan* p, const void* head, size_t cap, size_t* payload_size, uint64_t* changed,
                  bool accumulate)
{
    const EncScratch* st = static_cast<const EncScratch*>(head);
    *payload_size = st->total;
    if (st->n_spill || st->heap_top) p->overflow_seen = true;   // bodies past their slots: use the heap from now on
    if (changed) {
        const uint64_t* cnt = reinterpret_cast<const uint64_t*>(static_cast<const char*>(head) +
                                                                sizeof(EncScratch));
        if (accumulate)
            for (size_t i = 0; i < p->descs.size(); ++i) changed[i] += cnt[i];
        else
            memcpy(changed, cnt, p->descs.size() * 8);
    }
    if (st->err) return set_error(st->err, "dcr_encode: device error %d", st->err);
    if (st->total > cap)
        return set_error(DCR_ERR_CAPACITY, "dcr_encode: payload needs %llu bytes, capacity %zu",
                         (unsigned long long)st->total, cap);
    return DCR_OK;
}

int apply_result(dcr_recv_state* st, const ApplyScratch& a, dcr_apply_result* result)
{
    if (result) {
        result->target_version = a.target_version;
        result->n_frames = a.n_frames;
        result->frames_applied = a.applied;
        result->frames_skipped = a.skipped;
        result->pending = a.pending;
        result->window = a.window;
    }
    if (a.err) return set_error(a.err, "dcr_apply: device reported error %d", a.err);
    if (a.aborted) return set_error(DCR_ERR_ABORTED, "dcr_apply: injected fault stopped the apply");
    if (a.pending) return set_error(DCR_ERR_INCOMPLETE, "dcr_apply: %llu framed chunks not done",
                                    (unsigned long long)a.pending);
    if (a.target_version != st->pending) {
        std::fill(st->win_done.begin(), st->win_done.end(), 0);
        st->pending = a.target_version;
    }
    st->win_done[a.window] = 1;
    bool all = true;
    for (uint8_t d : st->win_done) all = all && d;
    if (all) {
        st->version = a.target_version;
        st->pending = ~0ull;
        if (result) result->committed = 1;
    }
    return DCR_OK;
}

}  // namespace dcr

static int apply_common(const dcr_plan* p, dcr_recv_state* st, const void* payload, size_t size,
                        void* target, uint64_t abort_at, uint32_t split, int retry_only,
                        dcr_apply_result* result, void* stream)
{
    if (result) memset(result, 0, sizeof(*result));
    if (!p || !st || !payload || !target) return set_error(DCR_ERR_INVALID, "dcr_apply: NULL argument");
    if (st->plan != p) return set_error(DCR_ERR_INVALID, "dcr_apply: state belongs to another plan");
    if (p->host_only) return set_error(DCR_ERR_INVALID, "dcr_apply: host-only plan");
    if (size < kStreamHdr) return set_error(DCR_ERR_CORRUPT, "dcr_apply: stream shorter than its header");
    if (!aligned16(payload) || !aligned16(target))
        return set_error(DCR_ERR_INVALID, "dcr_apply: payload/target not 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the first kernel and the commit check; the deferred-frame kernels only
    // when the first kernel deferred frames to them (a second status read)
    int rc = apply_launch_part(p, st, payload, size, target, abort_at, split, retry_only, kApplyFirst, s);
    if (rc) return rc;
    cudaError_t e = cudaMemcpyAsync(st->h_scratch, st->d_scratch, sizeof(ApplyScratch),
                                    cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_error(e, "dcr_apply status read");
    p->prof_deferred = false;
    if (st->h_scratch->hdr_ok && (st->h_scratch->n_defer || st->h_scratch->n_big)) {
        p->prof_deferred = true;
        rc = apply_launch_part(p, st, payload, size, target, abort_at, split, retry_only, kApplyDeferred, s);
        if (rc) return rc;
        e = cudaMemcpyAsync(st->h_scratch, st->d_scratch, sizeof(ApplyScratch), cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) return cuda_error(e, "dcr_apply status read");
    }
    if (p->profiling) {
        p->prof_apply_due = true;
        p->prof.apply_valid = 1;
        p->prof.apply_kernels = p->apply_kernels;
    }
    return apply_result(st, *st->h_scratch, result);
}

extern "C" int dcr_apply(const dcr_plan* p, dcr_recv_state* st, const void* payload, size_t size,
                         void* target, const dcr_fault* fault, dcr_apply_result* result, void* stream)
{
    uint64_t abort_at = fault ? fault->abort_after_frames : DCR_NO_FAULT;
    uint32_t split = fault ? fault->abort_split : 0;
    return apply_common(p, st, payload, size, target, abort_at, split, 0, result, stream);
}

extern "C" int dcr_apply_retry(const dcr_plan* p, dcr_recv_state* st, const void* payload, size_t size,
                               void* target, dcr_apply_result* result, void* stream)
{
    return apply_common(p, st, payload, size, target, DCR_NO_FAULT, 0, 1, result, stream);
}

extern "C" int dcr_plan_set_profiling(dcr_plan* p, int on)
{
    if (!p) return set_error(DCR_ERR_INVALID, "dcr_plan_set_profiling: NULL plan");
    if (p->host_only) return set_error(DCR_ERR_INVALID, "dcr_plan_set_profiling: host-only plan");
    if (on && !p->ev[0]) {
        for (cudaEvent_t& e : p->ev) {
            cudaError_t r = cudaEventCreate(&e);
            if (r != cudaSuccess) return cuda_error(r, "cudaEventCreate");
        }
    }
    p->profiling = on != 0;
    p->prof = dcr_profile{};
    p->prof_encode_due = p->prof_apply_due = false;
    return DCR_OK;
}

extern "C" int dcr_plan_last_profile(const dcr_plan* p, dcr_profile* out)
{
    if (!p || !out) return set_error(DCR_ERR_INVALID, "dcr_plan_last_profile: NULL argument");
    // the calls that recorded these events synchronised their stream
    if (p->prof_encode_due) {
        cudaEventElapsedTime(&p->prof.encode_ms, p->ev[0], p->ev[1]);
        cudaEventElapsedTime(&p->prof.finalize_ms, p->ev[1], p->ev[2]);
        p->prof_encode_due = false;
    }
    if (p->prof_apply_due) {
        cudaEventElapsedTime(&p->prof.apply_ms, p->ev[3], p->ev[4]);
        cudaEventElapsedTime(&p->prof.defer_ms, p->ev[p->prof_deferred ? 7 : 4], p->ev[5]);
        cudaEventElapsedTime(&p->prof.pending_ms, p->ev[5], p->ev[6]);
        p->prof_apply_due = false;
    }
    *out = p->prof;
    return DCR_OK;
}

extern "C" int dcr_dense_refit(const dcr_plan* p, const void* const* shards, void* target, void* stream)
{
    if (!p || !shards || !target) return set_error(DCR_ERR_INVALID, "dcr_dense_refit: NULL argument");
    if (p->host_only) return set_error(DCR_ERR_INVALID, "dcr_dense_refit: host-only plan");
    if (!aligned16(target)) return set_error(DCR_ERR_INVALID, "dcr_dense_refit: target not aligned");
    for (uint32_t r = 0; r < p->tp; ++r)
        if (p->shard_bytes[r] && (!shards[r] || !aligned16(shards[r])))
            return set_error(DCR_ERR_INVALID, "dcr_dense_refit: shard %u arena NULL or unaligned", r);
    return dense_launch(p, shards, target, static_cast<cudaStream_t>(stream));
}

// ---- ownership-sharded encode ----------------------------------------------
// (blog, "A strong baseline with the Blackwell-native DE": weight ownership
// is remapped so that the trainer ranks together cover the checkpoint
// exactly once, each rank compresses what it owns, and only the rank-local
// compressed payloads are gathered.)

namespace {

// Part `part` of `n_parts` of window w: the chunks whose first canonical
// byte falls in [part, part + 1) * B / n_parts, B = the window's bytes.
void part_range(const dcr_plan* p, uint32_t w, uint32_t part, uint32_t n_parts, uint64_t* begin, uint64_t* count)
{
    const uint64_t c0 = p->win_start[w], c1 = p->win_start[w + 1];
    const uint64_t s0 = p->chunk_start[c0], B = p->chunk_start[c1] - s0;
    auto first_at = [&](uint64_t q) {   // first chunk of the window starting at or after byte q
        const uint64_t t = s0 + (unsigned __int128)B * q / n_parts;
        return uint64_t(std::lower_bound(p->chunk_start.begin() + c0, p->chunk_start.begin() + c1, t) -
                        p->chunk_start.begin());
    };
    const uint64_t a = first_at(part), b = first_at(uint64_t(part) + 1);
    *begin = a;
    *count = b - a;
}

int part_args(const dcr_plan* p, uint32_t window, uint32_t part, uint32_t n_parts, const char* who)
{
    if (!p) return set_error(DCR_ERR_INVALID, "%s: NULL plan", who);
    if (window + 1 >= p->win_start.size()) return set_error(DCR_ERR_INVALID, "%s: window %u out of range", who, window);
    if (n_parts == 0 || n_parts > DCR_MAX_PARTS || part >= n_parts)
        return set_error(DCR_ERR_INVALID, "%s: part %u of %u (at most %u parts)", who, part, n_parts,
                         unsigned(DCR_MAX_PARTS));
    return DCR_OK;
}

}  // namespace

extern "C" int dcr_part_info_get(const dcr_plan* p, uint32_t window, uint32_t part, uint32_t n_parts,
                                 dcr_part_info* out)
{
    if (int rc = part_args(p, window, part, n_parts, "dcr_part_info_get")) return rc;
    if (!out) return set_error(DCR_ERR_INVALID, "dcr_part_info_get: NULL argument");
    memset(out, 0, sizeof(*out));
    part_range(p, window, part, n_parts, &out->chunk_begin, &out->chunk_count);
    out->canonical_bytes = p->chunk_start[out->chunk_begin + out->chunk_count] - p->chunk_start[out->chunk_begin];
    for (uint64_t c = out->chunk_begin; c < out->chunk_begin + out->chunk_count; ++c)
        out->shard_mask |= p->chunk_shards[c];
    return DCR_OK;
}

extern "C" int dcr_encode_part(const dcr_plan* p, uint32_t mode, uint32_t window, uint32_t part, uint32_t n_parts,
                               const void* const* olds, const void* const* news, dcr_part_size* size,
                               uint64_t* changed_per_tensor, void* stream)
{
    if (int rc = part_args(p, window, part, n_parts, "dcr_encode_part")) return rc;
    if (!olds || !news || !size) return set_error(DCR_ERR_INVALID, "dcr_encode_part: NULL argument");
    memset(size, 0, sizeof(*size));
    if (mode > DCR_MODE_OVERWRITE_ONLY) return set_error(DCR_ERR_INVALID, "dcr_encode_part: bad mode");
    if (p->host_only) return set_error(DCR_ERR_INVALID, "dcr_encode_part: host-only plan");
    p->part.valid = false;
    uint64_t cb, cc;
    part_range(p, window, part, n_parts, &cb, &cc);
    uint32_t need = 0;
    for (uint64_t c = cb; c < cb + cc; ++c) need |= p->chunk_shards[c];
    for (uint32_t r = 0; r < p->tp; ++r) {
        if ((need >> r & 1) && (!olds[r] || !news[r]))
            return set_error(DCR_ERR_INVALID, "dcr_encode_part: part %u reads shard %u, whose arena is NULL", part, r);
        if ((olds[r] && !aligned16(olds[r])) || (news[r] && !aligned16(news[r])))
            return set_error(DCR_ERR_INVALID, "dcr_encode_part: shard %u arena not 16-byte aligned", r);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = encode_size_launch(p, mode, cb, cc, olds, news, s);
    if (rc) return rc;
    cudaError_t e = cudaMemcpyAsync(p->h_enc, p->d_enc, p->enc_head_bytes, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_error(e, "dcr_encode_part status read");
    const EncScratch* hs = static_cast<const EncScratch*>(p->h_enc);
    if (hs->n_spill || hs->heap_top) p->overflow_seen = true;
    if (changed_per_tensor)
        memcpy(changed_per_tensor, static_cast<const char*>(p->h_enc) + sizeof(EncScratch), p->descs.size() * 8);
    if (hs->err) return set_error(hs->err, "dcr_encode_part: device error %d", hs->err);
    size->n_frames = hs->n_frames;
    size->frame_bytes = hs->total - kStreamHdr - 8 * hs->n_frames;
    p->part.valid = true;
    p->part.mode = mode;
    p->part.window = window;
    p->part.chunk_begin = cb;
    p->part.chunk_count = cc;
    p->part.frame_bytes = size->frame_bytes;
    p->part.n_frames = size->n_frames;
    for (uint32_t r = 0; r < DCR_MAX_TP; ++r) {
        p->part.olds[r] = r < p->tp ? olds[r] : nullptr;
        p->part.news[r] = r < p->tp ? news[r] : nullptr;
    }
    return DCR_OK;
}

extern "C" int dcr_encode_part_write(const dcr_plan* p, uint64_t frame_offset, void* frames, size_t frames_cap,
                                     void* index, void* stream)
{
    if (!p) return set_error(DCR_ERR_INVALID, "dcr_encode_part_write: NULL plan");
    if (!p->part.valid)
        return set_error(DCR_ERR_INVALID, "dcr_encode_part_write: no part sized by dcr_encode_part on this plan");
    if ((p->part.frame_bytes && !frames) || (p->part.n_frames && !index))
        return set_error(DCR_ERR_INVALID, "dcr_encode_part_write: NULL buffer");
    if (frames_cap < p->part.frame_bytes)
        return set_error(DCR_ERR_CAPACITY, "dcr_encode_part_write: frames need %llu bytes, capacity %zu",
                         (unsigned long long)p->part.frame_bytes, frames_cap);
    if ((frames && !aligned16(frames)) || (reinterpret_cast<uintptr_t>(index) & 7) || frame_offset % 16)
        return set_error(DCR_ERR_INVALID, "dcr_encode_part_write: frames / frame_offset not 16-byte aligned, "
                                          "or index not 8-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int rc = encode_write_launch(p, p->part.mode, p->part.chunk_begin, p->part.chunk_count, p->part.olds,
                                 p->part.news, static_cast<uint8_t*>(frames), frame_offset,
                                 static_cast<uint64_t*>(index), s);
    if (rc) return rc;
    cudaError_t e = cudaMemcpyAsync(p->h_enc, p->d_enc, p->enc_head_bytes, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_error(e, "dcr_encode_part_write status read");
    const EncScratch* hs = static_cast<const EncScratch*>(p->h_enc);
    if (hs->err) return set_error(hs->err, "dcr_encode_part_write: device error %d", hs->err);
    return DCR_OK;
}

extern "C" int dcr_stream_layout(uint32_t n_parts, const dcr_part_size* sizes, uint64_t* frame_offsets,
                                 uint64_t* index_offsets, uint64_t* total)
{
    if (n_parts == 0 || n_parts > DCR_MAX_PARTS || !sizes || !frame_offsets || !index_offsets || !total)
        return set_error(DCR_ERR_INVALID, "dcr_stream_layout: bad arguments");
    uint64_t F = 0, NF = 0;
    for (uint32_t q = 0; q < n_parts; ++q) {
        if (sizes[q].frame_bytes % 16) return set_error(DCR_ERR_INVALID, "dcr_stream_layout: part %u frame bytes "
                                                                          "not a multiple of 16", q);
        frame_offsets[q] = kStreamHdr + F;
        F += sizes[q].frame_bytes;
        NF += sizes[q].n_frames;
    }
    uint64_t idx = kStreamHdr + F;
    for (uint32_t q = 0; q < n_parts; ++q) {
        index_offsets[q] = idx;
        idx += 8 * sizes[q].n_frames;
    }
    *total = idx;
    return DCR_OK;
}

extern "C" int dcr_stream_header(const dcr_plan* p, uint32_t mode, uint32_t window, uint64_t base_version,
                                 uint64_t target_version, uint64_t n_frames, uint64_t frame_bytes, void* header)
{
    if (!p || !header) return set_error(DCR_ERR_INVALID, "dcr_stream_header: NULL argument");
    if (mode > DCR_MODE_OVERWRITE_ONLY) return set_error(DCR_ERR_INVALID, "dcr_stream_header: bad mode");
    if (window + 1 >= p->win_start.size())
        return set_error(DCR_ERR_INVALID, "dcr_stream_header: window %u out of range", window);
    if (frame_bytes % 16) return set_error(DCR_ERR_INVALID, "dcr_stream_header: frame bytes not a multiple of 16");
    uint8_t* h = static_cast<uint8_t*>(header);
    auto put32 = [&](int at, uint32_t v) { for (int i = 0; i < 4; ++i) h[at + i] = uint8_t(v >> (8 * i)); };
    auto put64 = [&](int at, uint64_t v) { put32(at, uint32_t(v)); put32(at + 4, uint32_t(v >> 32)); };
    put32(0, kStreamMagic);
    put32(4, kFormat);
    put64(8, p->hash);
    put64(16, base_version);
    put64(24, target_version);
    put32(32, window);
    put32(36, mode == DCR_MODE_OVERWRITE_ONLY ? kStreamOverwriteOnly : 0u);
    put32(40, uint32_t(p->win_start[window]));
    put32(44, uint32_t(p->win_start[window + 1] - p->win_start[window]));
    put64(48, n_frames);
    put64(56, kStreamHdr + frame_bytes + 8 * n_frames);
    return DCR_OK;
}

// ---- overwrite-only retry from the XOR stream -------------------------------
extern "C" int dcr_encode_retry(const dcr_plan* p, const void* xor_payload, size_t xor_size,
                                const void* const* news, void* payload, size_t cap, size_t* payload_size,
                                void* stream)
{
    if (!p || !xor_payload || !news || !payload_size)
        return set_error(DCR_ERR_INVALID, "dcr_encode_retry: NULL argument");
    *payload_size = 0;
    if (p->host_only) return set_error(DCR_ERR_INVALID, "dcr_encode_retry: host-only plan");
    if (xor_size < kStreamHdr) return set_error(DCR_ERR_CORRUPT, "dcr_encode_retry: stream shorter than its header");
    if (!aligned16(xor_payload) || (payload && !aligned16(payload)))
        return set_error(DCR_ERR_INVALID, "dcr_encode_retry: stream or payload not 16-byte aligned");
    for (uint32_t r = 0; r < p->tp; ++r) {
        if (p->shard_bytes[r] && !news[r])
            return set_error(DCR_ERR_INVALID, "dcr_encode_retry: shard %u arena is NULL", r);
        if (news[r] && !aligned16(news[r]))
            return set_error(DCR_ERR_INVALID, "dcr_encode_retry: shard %u arena not 16-byte aligned", r);
    }
    p->part.valid = false;   // the plan's scratch now holds this encode
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t h[64];
    cudaError_t e = cudaMemcpyAsync(h, xor_payload, sizeof(h), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_error(e, "dcr_encode_retry header read");
    auto u32 = [&](int at) { uint32_t v; memcpy(&v, h + at, 4); return v; };
    auto u64 = [&](int at) { uint64_t v; memcpy(&v, h + at, 8); return v; };
    const uint64_t total = u64(56), nf = u64(48), window = u32(32);
    if (u32(0) != kStreamMagic || u32(4) != kFormat || total > xor_size || total < kStreamHdr || total % 8 ||
        nf > (total - kStreamHdr) / 8)
        return set_error(DCR_ERR_CORRUPT, "dcr_encode_retry: malformed stream header");
    if (u64(8) != p->hash || window + 1 >= p->win_start.size() || u32(40) != p->win_start[window] ||
        u32(44) != p->win_start[window + 1] - p->win_start[window])
        return set_error(DCR_ERR_INVALID, "dcr_encode_retry: stream of another plan or window");
    int rc = retry_launch(p, xor_payload, total - 8 * nf, nf, uint32_t(window), u64(16), u64(24), news, payload,
                          payload ? cap : 0, s);
    if (rc) return rc;
    e = cudaMemcpyAsync(p->h_enc, p->d_enc, p->enc_head_bytes, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_error(e, "dcr_encode_retry status read");
    if (p->profiling) {
        p->prof_encode_due = true;
        p->prof.encode_valid = 1;
        p->prof.encode_kernels = kRetryKernels;
    }
    const EncScratch* hs = static_cast<const EncScratch*>(p->h_enc);
    *payload_size = hs->total;
    if (hs->err) return set_error(hs->err, "dcr_encode_retry: device error %d", hs->err);
    if (hs->total > (payload ? cap : 0))
        return set_error(DCR_ERR_CAPACITY, "dcr_encode_retry: payload needs %llu bytes, capacity %zu",
                         (unsigned long long)hs->total, payload ? cap : size_t(0));
    return DCR_OK;
}
