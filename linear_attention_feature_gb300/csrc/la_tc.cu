// Selection between the tensor-core forward kernels.
#include <cstdint>

#include "la_tc.h"

namespace la {

static bool aligned16(const void *p) {
    return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

bool tc_supported(const FwdShape &sh, la_dtype dtype, int causal,
                  const void *q, const void *k, const void *v,
                  const void *out) {
    if (dtype != LA_BF16) return false;
    if (sh.d != 64 && sh.d != 128) return false;
    (void)causal;
    return aligned16(q) && aligned16(k) && aligned16(v) && aligned16(out);
}

TcResult tc_forward(const void *q, const void *k, const void *v, void *out,
                    const FwdShape &sh, int causal, const DecayArgs &dk,
                    int segment_chunks, int *status, void *ws, size_t ws_bytes,
                    float *S_out, float *z_out, const float *gates,
                    cudaStream_t stream) {
    if (causal)
        return launch_causal_tc(q, k, v, out, sh, dk, segment_chunks, status,
                                ws, ws_bytes, S_out, z_out, gates, stream);
    return launch_noncausal_tc(q, k, v, out, sh, segment_chunks, status, ws,
                               ws_bytes, stream);
}

size_t tc_workspace_bytes(const FwdShape &sh, int causal, bool decay,
                          int segment_chunks, int sms) {
    if (sh.BH() == 0 || sh.N == 0) return 0;
    return causal ? causal_tc_workspace_bytes(sh, decay, segment_chunks, sms)
                  : noncausal_tc_workspace_bytes(sh, segment_chunks, sms);
}

namespace {

__global__ void zero_words_kernel(uint4 *p, size_t n) {
    // the forward kernel after this one may start its prologue now; it waits
    // for this kernel's completion before it reads the cleared words
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        p[i] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace

namespace {
thread_local long long t_debug_wait = 0;
thread_local int t_debug_hold = -1;
thread_local int t_debug_fail_allocs = 0;
}  // namespace

void tc_debug_set_timeout(long long wait_cycles, int hold_segment) {
    t_debug_wait = wait_cycles;
    t_debug_hold = hold_segment;
}

bool tc_debug_take_timeout(long long *wait_cycles, int *hold_segment) {
    if (t_debug_wait <= 0) return false;
    *wait_cycles = t_debug_wait;
    *hold_segment = t_debug_hold;
    t_debug_wait = 0;
    t_debug_hold = -1;
    return true;
}

void tc_debug_fail_allocs(int n) { t_debug_fail_allocs = n > 0 ? n : 0; }

cudaError_t tc_workspace_alloc(void **ws, size_t bytes, cudaStream_t stream) {
    if (t_debug_fail_allocs > 0) {
        --t_debug_fail_allocs;
        return cudaErrorMemoryAllocation;
    }
    return cudaMallocAsync(ws, bytes, stream);
}

cudaError_t tc_zero_words(void *p, size_t bytes, cudaStream_t stream) {
    const size_t n = bytes / 16;
    if (n == 0) return cudaSuccess;
    const size_t want = (n + 255) / 256;
    const int blocks = (int)(want < 152 ? want : 152);
    zero_words_kernel<<<blocks, 256, 0, stream>>>(static_cast<uint4 *>(p), n);
    return cudaGetLastError();
}

}  // namespace la
