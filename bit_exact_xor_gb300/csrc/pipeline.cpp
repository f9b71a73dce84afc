// Pipelined refit of a whole model through host memory: the window-by-window
// encode -> transfer -> apply of dcr_encode + dcr_apply, with the transfer of
// one window overlapping the compute of its neighbours.
//
// Method: NeMo-DCR paper summary, "Pipelined transfer" (a window's stream is
// built while the previous one is sent, so build and transfer overlap) and
// the popular write-up's transfer step.  Here the wire is pinned host memory:
// each window's stream goes device -> host -> device before it is applied.
//
// Schedule on the caller's stream S (kernels) and a copy stream C, with two
// buffers of each kind (slot k & 1):
//
//   S: encode(0) encode(1) apply(0) encode(2) apply(1) encode(3) apply(2) ...
//   C:           D2H+H2D(0)         D2H+H2D(1)         D2H+H2D(2) ...
//
// The host learns window k's stream size from its status (read back in
// stream order right after its kernels) before it issues the copies; the
// next encode into a buffer waits for that buffer's D2H, a copy into a
// receive buffer waits for the apply that read it, and an apply waits for
// its H2D.  Apply statuses are checked in window order, one window behind.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "dcr_internal.h"

using namespace dcr;

namespace dcr {

void pipe_release(const dcr_plan* p)
{
    for (cudaEvent_t& e : p->pipe_ev) {
        if (e) cudaEventDestroy(e);
        e = nullptr;
    }
    if (p->pipe_copy) cudaStreamDestroy(p->pipe_copy);
    p->pipe_copy = nullptr;
}

}  // namespace dcr

namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// largest payload bound over the plan's windows
size_t max_window_bound(const dcr_plan* p)
{
    size_t best = 0;
    for (size_t w = 0; w + 1 < p->win_start.size(); ++w) {
        dcr_window_info wi;
        if (dcr_window_info_get(p, uint32_t(w), &wi) == DCR_OK && wi.payload_bound > best)
            best = size_t(wi.payload_bound);
    }
    return best;
}

struct Layout {
    size_t bound;                      // one stream buffer
    size_t dev_bytes, host_bytes;
    size_t h_enc_off[2], h_app_off[2]; // status mirrors in host_buf, after the two staging buffers
};

Layout layout_of(const dcr_plan* p)
{
    Layout L{};
    L.bound = round_up(max_window_bound(p));
    L.dev_bytes = 4 * L.bound;         // two send buffers, two receive buffers
    size_t off = 2 * L.bound;          // two host staging buffers
    for (int i = 0; i < 2; ++i) {
        L.h_enc_off[i] = off;
        off += round_up(p->enc_head_bytes);
    }
    for (int i = 0; i < 2; ++i) {
        L.h_app_off[i] = off;
        off += round_up(sizeof(ApplyScratch));
    }
    L.host_bytes = off;
    return L;
}

bool aligned(const void* q, size_t a) { return (reinterpret_cast<uintptr_t>(q) % a) == 0; }

// the copy stream and events, created on the first pipelined call and kept
// with the plan (released by dcr_plan_destroy)
cudaError_t pipe_objects(const dcr_plan* p)
{
    if (p->pipe_copy) return cudaSuccess;
    cudaError_t e = cudaStreamCreateWithFlags(&p->pipe_copy, cudaStreamNonBlocking);
    for (int i = 0; i < 8 && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&p->pipe_ev[i], cudaEventDisableTiming);
    if (e != cudaSuccess) pipe_release(p);
    return e;
}

}  // namespace

extern "C" int dcr_pipeline_sizes(const dcr_plan* p, size_t* device_bytes, size_t* host_bytes)
{
    if (!p || !device_bytes || !host_bytes) return set_error(DCR_ERR_INVALID, "dcr_pipeline_sizes: NULL argument");
    const Layout L = layout_of(p);
    *device_bytes = L.dev_bytes;
    *host_bytes = L.host_bytes;
    return DCR_OK;
}

extern "C" int dcr_refit_pipelined(const dcr_plan* p, dcr_recv_state* st, uint32_t mode,
                                   const void* const* olds, const void* const* news, uint64_t base_version,
                                   uint64_t target_version, void* target, void* device_buf, size_t device_bytes,
                                   void* host_buf, size_t host_bytes, uint64_t* changed_per_tensor,
                                   dcr_pipeline_stats* stats, void* stream)
{
    if (stats) memset(stats, 0, sizeof(*stats));
    if (!p || !st || !olds || !news || !target || !device_buf || !host_buf)
        return set_error(DCR_ERR_INVALID, "dcr_refit_pipelined: NULL argument");
    if (st->plan != p) return set_error(DCR_ERR_INVALID, "dcr_refit_pipelined: state belongs to another plan");
    if (mode > DCR_MODE_OVERWRITE_ONLY) return set_error(DCR_ERR_INVALID, "dcr_refit_pipelined: bad mode");
    if (p->host_only) return set_error(DCR_ERR_INVALID, "dcr_refit_pipelined: host-only plan");
    p->part.valid = false;   // the plan's scratch now holds these encodes
    const Layout L = layout_of(p);
    if (device_bytes < L.dev_bytes || host_bytes < L.host_bytes)
        return set_error(DCR_ERR_INVALID, "dcr_refit_pipelined: buffers too small (need %zu device, %zu host bytes)",
                         L.dev_bytes, L.host_bytes);
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, host_buf) != cudaSuccess || attr.type != cudaMemoryTypeHost) {
        cudaGetLastError();
        return set_error(DCR_ERR_INVALID, "dcr_refit_pipelined: host_buf is not pinned host memory");
    }
    if (!aligned(device_buf, kAlign) || !aligned(host_buf, kAlign) || !aligned(target, 16))
        return set_error(DCR_ERR_INVALID, "dcr_refit_pipelined: buffers not aligned");
    for (uint32_t r = 0; r < p->tp; ++r) {
        if (p->shard_bytes[r] && (!olds[r] || !news[r]))
            return set_error(DCR_ERR_INVALID, "dcr_refit_pipelined: shard %u arena is NULL", r);
        if ((olds[r] && !aligned(olds[r], 16)) || (news[r] && !aligned(news[r], 16)))
            return set_error(DCR_ERR_INVALID, "dcr_refit_pipelined: shard %u arena not 16-byte aligned", r);
    }
    if (changed_per_tensor) memset(changed_per_tensor, 0, p->descs.size() * 8);

    cudaError_t e = pipe_objects(p);
    if (e != cudaSuccess) return cuda_error(e, "dcr_refit_pipelined: stream/event creation");
    struct {
        cudaStream_t copy;
        cudaEvent_t *enc, *d2h, *h2d, *app;
    } R{p->pipe_copy, p->pipe_ev, p->pipe_ev + 2, p->pipe_ev + 4, p->pipe_ev + 6};
    cudaStream_t S = static_cast<cudaStream_t>(stream);
    uint8_t* dev = static_cast<uint8_t*>(device_buf);
    uint8_t* host = static_cast<uint8_t*>(host_buf);
    uint8_t* send[2] = {dev, dev + L.bound};
    uint8_t* recv[2] = {dev + 2 * L.bound, dev + 3 * L.bound};
    uint8_t* stage[2] = {host, host + L.bound};
    void* h_enc[2] = {host + L.h_enc_off[0], host + L.h_enc_off[1]};
    ApplyScratch* h_app[2] = {reinterpret_cast<ApplyScratch*>(host + L.h_app_off[0]),
                              reinterpret_cast<ApplyScratch*>(host + L.h_app_off[1])};
    const uint32_t W = uint32_t(p->win_start.size() - 1);
    const int retry_only = mode == DCR_MODE_OVERWRITE_ONLY;

    int rc = DCR_OK;
    uint32_t launched_apply = 0;   // applies issued; their statuses are checked in order
    uint32_t checked_apply = 0;
    uint64_t total = 0, biggest = 0;
    bool committed = false;

    auto launch_encode = [&](uint32_t k) -> int {
        const int s = int(k & 1);
        if (k >= 2) {   // the send buffer's previous stream has left for the host
            cudaError_t x = cudaStreamWaitEvent(S, R.d2h[s], 0);
            if (x != cudaSuccess) return cuda_error(x, "dcr_refit_pipelined: wait");
        }
        int r = encode_launch(p, mode, k, olds, news, base_version, target_version, send[s], L.bound, S);
        if (r) return r;
        cudaError_t x = cudaMemcpyAsync(h_enc[s], p->d_enc, p->enc_head_bytes, cudaMemcpyDeviceToHost, S);
        if (x == cudaSuccess) x = cudaEventRecord(R.enc[s], S);
        return x == cudaSuccess ? DCR_OK : cuda_error(x, "dcr_refit_pipelined: encode status");
    };
    auto check_apply = [&]() -> int {   // the oldest unchecked apply
        const int s = int(checked_apply & 1);
        cudaError_t x = cudaEventSynchronize(R.app[s]);
        if (x != cudaSuccess) return cuda_error(x, "dcr_refit_pipelined: apply status");
        dcr_apply_result res;
        memset(&res, 0, sizeof(res));
        const int r = apply_result(st, *h_app[s], &res);
        ++checked_apply;
        committed = committed || res.committed;
        return r;
    };

    if (W > 0) rc = launch_encode(0);
    for (uint32_t k = 0; k < W && rc == DCR_OK; ++k) {
        const int s = int(k & 1);
        if (k + 1 < W && (rc = launch_encode(k + 1)) != DCR_OK) break;
        // window k's stream size, from its status
        if ((e = cudaEventSynchronize(R.enc[s])) != cudaSuccess) {
            rc = cuda_error(e, "dcr_refit_pipelined: encode status");
            break;
        }
        size_t size = 0;
        if ((rc = encode_result(p, h_enc[s], L.bound, &size, changed_per_tensor, true)) != DCR_OK) break;
        total += size;
        if (size > biggest) biggest = size;
        // the transfer, on the copy stream: after the encode, and after the
        // apply that last read this receive buffer
        e = cudaStreamWaitEvent(R.copy, R.enc[s], 0);
        if (e == cudaSuccess && k >= 2) e = cudaStreamWaitEvent(R.copy, R.app[s], 0);
        if (e == cudaSuccess) e = cudaMemcpyAsync(stage[s], send[s], size, cudaMemcpyDeviceToHost, R.copy);
        if (e == cudaSuccess) e = cudaEventRecord(R.d2h[s], R.copy);
        if (e == cudaSuccess) e = cudaMemcpyAsync(recv[s], stage[s], size, cudaMemcpyHostToDevice, R.copy);
        if (e == cudaSuccess) e = cudaEventRecord(R.h2d[s], R.copy);
        // the apply, on the kernel stream once the stream has arrived
        if (e == cudaSuccess) e = cudaStreamWaitEvent(S, R.h2d[s], 0);
        if (e != cudaSuccess) {
            rc = cuda_error(e, "dcr_refit_pipelined: transfer");
            break;
        }
        // a window's status mirror is reused two windows on: check the
        // previous window's apply before this one can overwrite slot k ^ 1's
        if (launched_apply > checked_apply + 1 && (rc = check_apply()) != DCR_OK) break;
        if ((rc = apply_launch(p, st, recv[s], size, target, DCR_NO_FAULT, 0, retry_only, S)) != DCR_OK) break;
        e = cudaMemcpyAsync(h_app[s], st->d_scratch, sizeof(ApplyScratch), cudaMemcpyDeviceToHost, S);
        if (e == cudaSuccess) e = cudaEventRecord(R.app[s], S);
        if (e != cudaSuccess) {
            rc = cuda_error(e, "dcr_refit_pipelined: apply status");
            break;
        }
        ++launched_apply;
        if (launched_apply > checked_apply + 1 && (rc = check_apply()) != DCR_OK) break;
    }
    while (rc == DCR_OK && checked_apply < launched_apply) rc = check_apply();
    // whatever is still in flight finishes before the buffers go back to the caller
    cudaError_t e1 = cudaStreamSynchronize(S);
    cudaError_t e2 = cudaStreamSynchronize(R.copy);
    if (rc == DCR_OK && (e1 != cudaSuccess || e2 != cudaSuccess))
        rc = cuda_error(e1 != cudaSuccess ? e1 : e2, "dcr_refit_pipelined: drain");
    if (stats) {
        stats->windows = checked_apply;
        stats->payload_bytes = total;
        stats->max_window_payload = biggest;
        stats->committed = committed ? 1u : 0u;
    }
    return rc;
}
