// la_forward_host: la_forward on host buffers.  The host-to-device copies,
// the kernels and the device-to-host copies run over groups of heads on
// three streams, so that group g+1 is copied in while group g computes and
// group g-1 is copied out.  The contract is in include/linattn.h.
#include <algorithm>
#include <cstdio>
#include <mutex>

#include "la_internal.h"

namespace la {
namespace {

constexpr int kMaxDevices = 64;
// Measured on GB300 (NVLink-C2C, ~210 GB/s host to device): four groups
// already hide the kernels behind the copies; more groups only add copy
// operations, and the device-to-host copies slow the host-to-device ones.
constexpr int kMaxGroups = 4;
// Events per device: one start, one end, and per group "inputs copied" and
// "group computed".
constexpr int kEvents = 2 + 2 * kMaxGroups;

struct CopyEngine {
    bool ready = false;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t ev[kEvents] = {};
};

std::mutex g_host_mu[kMaxDevices];
CopyEngine g_engine[kMaxDevices];

thread_local char g_host_err[256];

la_status host_fail(la_status s, const char *msg) {
    set_last_error(msg);
    return s;
}

la_status host_cuda_fail(cudaError_t e, const char *where) {
    std::snprintf(g_host_err, sizeof(g_host_err), "%s: %s", where,
                  cudaGetErrorString(e));
    set_last_error(g_host_err);
    return LA_ERR_CUDA;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// One tensor's bytes in the workspace (each of q, k, v, out starts on a
// 256-byte boundary).
size_t tensor_bytes(long long BH, int N, int d, la_dtype dtype) {
    const size_t elem = dtype == LA_BF16 ? 2 : 4;
    return round_up((size_t)BH * (size_t)N * (size_t)d * elem, 256);
}

// The copy streams and events of the current device, created on first use
// (the caller holds g_host_mu[dev]).
cudaError_t engine_of(int dev, CopyEngine **out) {
    CopyEngine &en = g_engine[dev];
    if (!en.ready) {
        cudaError_t e;
        if ((e = cudaStreamCreateWithFlags(&en.in, cudaStreamNonBlocking)) != cudaSuccess)
            return e;
        if ((e = cudaStreamCreateWithFlags(&en.out, cudaStreamNonBlocking)) != cudaSuccess)
            return e;
        for (int i = 0; i < kEvents; ++i)
            if ((e = cudaEventCreateWithFlags(&en.ev[i], cudaEventDisableTiming)) != cudaSuccess)
                return e;
        en.ready = true;
    }
    *out = &en;
    return cudaSuccess;
}

// A group: heads [b0, b0 + nb) x [h0, h0 + nh) of the [B][H] grid, stored
// contiguously (whole batches, or a range of heads inside one batch).
struct Group {
    int b0, nb, h0, nh;
};

// At most kMaxGroups groups of at least ~8 MiB of input each.
int make_groups(int B, int H, long long in_bytes, Group *g) {
    const int want = (int)std::min<long long>(kMaxGroups, std::max<long long>(1, in_bytes >> 23));
    int n = 0;
    if (B >= want) {
        const int nb = (B + want - 1) / want;
        for (int b = 0; b < B; b += nb) g[n++] = {b, std::min(nb, B - b), 0, H};
    } else {
        // B * split <= want groups, each a range of heads of one batch
        const int split = std::max(1, std::min(H, want / B));
        const int nh = (H + split - 1) / split;
        for (int b = 0; b < B; ++b)
            for (int h = 0; h < H; h += nh) g[n++] = {b, 1, h, std::min(nh, H - h)};
    }
    return n;
}

// Kernel scratch for the largest group, over every variant of the call (so
// that one size serves causal or not, with or without decay).
size_t group_scratch_bytes(int B, int H, int N, int d, la_dtype dtype) {
    Group gr[kMaxGroups];
    const size_t elem = dtype == LA_BF16 ? 2 : 4;
    const int ng = make_groups(B, H, 3LL * B * H * N * d * (long long)elem, gr);
    size_t need = 0;
    for (int i = 0; i < ng; ++i)
        for (int causal = 0; causal < 2; ++causal)
            for (int dec = 0; dec < 2; ++dec)
                need = std::max(need, forward_workspace_bytes(gr[i].nb, gr[i].nh, N, d, causal,
                                                              dec != 0, dtype));
    return round_up(need, 256);
}

// After a failure part-way through: `stream` still waits for whatever copies
// were enqueued, so that the caller's buffers are not reused under them.
void join_copies(CopyEngine *en, cudaStream_t s) {
    cudaEventRecord(en->ev[1], en->in);
    cudaStreamWaitEvent(s, en->ev[1], 0);
    cudaEventRecord(en->ev[1], en->out);
    cudaStreamWaitEvent(s, en->ev[1], 0);
}

}  // namespace
}  // namespace la

using namespace la;

extern "C" {

__attribute__((visibility("default")))
size_t la_forward_host_workspace_bytes(int B, int H, int N, int d, la_dtype dtype) {
    if (B < 0 || H < 0 || N < 0 || d < 1 || d > LA_MAX_D) return 0;
    if (dtype != LA_F32 && dtype != LA_BF16) return 0;
    if ((long long)B * H == 0 || N == 0) return 0;
    return 4 * tensor_bytes((long long)B * H, N, d, dtype) +
           group_scratch_bytes(B, H, N, d, dtype);
}

__attribute__((visibility("default")))
la_status la_forward_host(const void *q, const void *k, const void *v,
                          void *out, int B, int H, int N, int d, int causal,
                          const float *decay, la_dtype dtype, void *workspace,
                          size_t workspace_bytes, la_stream_t stream) {
    if (!q || !k || !v || !out)
        return host_fail(LA_ERR_INVALID_ARG, "la_forward_host: null host pointer");
    if (B < 0 || H < 0 || N < 0)
        return host_fail(LA_ERR_INVALID_ARG, "la_forward_host: negative B, H or N");
    if (d < 1 || d > LA_MAX_D)
        return host_fail(LA_ERR_INVALID_ARG, "la_forward_host: d must be in 1..256");
    if (dtype != LA_F32 && dtype != LA_BF16)
        return host_fail(LA_ERR_INVALID_ARG, "la_forward_host: unknown dtype");
    if (causal != 0 && causal != 1)
        return host_fail(LA_ERR_INVALID_ARG, "la_forward_host: causal must be 0 or 1");
    if (out == q || out == k || out == v)
        return host_fail(LA_ERR_INVALID_ARG, "la_forward_host: out aliases an input");
    if (decay && !causal)
        return host_fail(LA_ERR_INVALID_ARG,
                         "la_forward_host: decay is defined for the causal form only");
    if (decay && H > LA_MAX_DECAY_HEADS)
        return host_fail(LA_ERR_UNSUPPORTED,
                         "la_forward_host: decay given for more than 1024 heads");
    if (decay)
        for (int h = 0; h < H; ++h)
            if (!(decay[h] >= 0.f && decay[h] <= 1.f))
                return host_fail(LA_ERR_INVALID_ARG,
                                 "la_forward_host: decay values must lie in [0, 1]");
    const long long BH = (long long)B * H;
    if (BH == 0 || N == 0) return LA_OK;
    const size_t tb = tensor_bytes(BH, N, d, dtype);
    const size_t scratch_bytes = group_scratch_bytes(B, H, N, d, dtype);
    if (!workspace || workspace_bytes < 4 * tb + scratch_bytes)
        return host_fail(LA_ERR_INVALID_ARG,
                         "la_forward_host: workspace missing or smaller than "
                         "la_forward_host_workspace_bytes()");
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0)
        return host_fail(LA_ERR_INVALID_ARG,
                         "la_forward_host: workspace must be 256-byte aligned");

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return host_cuda_fail(e, "la_forward_host: device query");
    if (dev < 0 || dev >= kMaxDevices)
        return host_fail(LA_ERR_UNSUPPORTED, "la_forward_host: device index");
    std::lock_guard<std::mutex> lk(g_host_mu[dev]);
    CopyEngine *en = nullptr;
    if ((e = engine_of(dev, &en)) != cudaSuccess)
        return host_cuda_fail(e, "la_forward_host: copy streams");

    const size_t elem = dtype == LA_BF16 ? 2 : 4;
    const size_t head_bytes = (size_t)N * d * elem;
    char *dq = static_cast<char *>(workspace);
    char *dk = dq + tb, *dv = dk + tb, *dout = dv + tb;
    // the groups' kernels run one after another on `stream`, so they share
    // one kernel scratch (no allocation between the copies)
    char *scratch = dout + tb;
    const char *hq = static_cast<const char *>(q), *hk = static_cast<const char *>(k),
               *hv = static_cast<const char *>(v);
    char *hout = static_cast<char *>(out);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

    Group gr[kMaxGroups];
    const int ng = make_groups(B, H, 3 * (long long)BH * (long long)head_bytes, gr);
    cudaEvent_t ev_start = en->ev[0], ev_end = en->ev[1];
    // copies start after the work already on `stream` (earlier users of
    // the workspace and of the host buffers)
    if ((e = cudaEventRecord(ev_start, s)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(en->in, ev_start, 0)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(en->out, ev_start, 0)) != cudaSuccess)
        return host_cuda_fail(e, "la_forward_host: ordering after the stream");
    // every input copy first, so that the copy engine never waits for the
    // host to enqueue a group's kernels
    for (int i = 0; i < ng; ++i) {
        const Group &g = gr[i];
        const size_t off = ((size_t)g.b0 * H + g.h0) * head_bytes;
        const size_t bytes = (size_t)g.nb * g.nh * head_bytes;
        if ((e = cudaMemcpyAsync(dq + off, hq + off, bytes, cudaMemcpyHostToDevice, en->in)) != cudaSuccess ||
            (e = cudaMemcpyAsync(dk + off, hk + off, bytes, cudaMemcpyHostToDevice, en->in)) != cudaSuccess ||
            (e = cudaMemcpyAsync(dv + off, hv + off, bytes, cudaMemcpyHostToDevice, en->in)) != cudaSuccess ||
            (e = cudaEventRecord(en->ev[2 + 2 * i], en->in)) != cudaSuccess) {
            join_copies(en, s);
            return host_cuda_fail(e, "la_forward_host: input copy");
        }
    }
    // then per group: its kernels once its inputs are in, its output copy
    // once its kernels are done
    for (int i = 0; i < ng; ++i) {
        const Group &g = gr[i];
        const size_t off = ((size_t)g.b0 * H + g.h0) * head_bytes;
        const size_t bytes = (size_t)g.nb * g.nh * head_bytes;
        cudaEvent_t ev_in = en->ev[2 + 2 * i], ev_done = en->ev[3 + 2 * i];
        if ((e = cudaStreamWaitEvent(s, ev_in, 0)) != cudaSuccess) {
            join_copies(en, s);
            return host_cuda_fail(e, "la_forward_host: input copy");
        }
        const la_status st = forward_with_workspace(
            dq + off, dk + off, dv + off, dout + off, g.nb, g.nh, N, d, causal,
            decay ? decay + g.h0 : nullptr, dtype, 0, 0,
            scratch_bytes ? scratch : nullptr, scratch_bytes, nullptr, nullptr,
            nullptr, nullptr, stream);
        if (st != LA_OK) {
            join_copies(en, s);
            return st;
        }
        if ((e = cudaEventRecord(ev_done, s)) != cudaSuccess ||
            (e = cudaStreamWaitEvent(en->out, ev_done, 0)) != cudaSuccess ||
            (e = cudaMemcpyAsync(hout + off, dout + off, bytes, cudaMemcpyDeviceToHost, en->out)) != cudaSuccess) {
            join_copies(en, s);
            return host_cuda_fail(e, "la_forward_host: output copy");
        }
    }
    // `stream` continues once the last output copy is done
    if ((e = cudaEventRecord(ev_end, en->out)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s, ev_end, 0)) != cudaSuccess)
        return host_cuda_fail(e, "la_forward_host: ordering before the stream");
    return LA_OK;
}

}  // extern "C"
