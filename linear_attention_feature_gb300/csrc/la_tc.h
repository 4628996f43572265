// Tensor-core (tcgen05 + TMEM + TMA) forward kernels: selection and launch.
#pragma once

#include "la_internal.h"

namespace la {

struct TcResult {
    la_status status;
    cudaError_t cuda;
    const char *where;
};

// True when the tensor-core kernels take this problem: bf16, d in {64, 128},
// all four tensors 16-byte aligned (a TMA requirement).
bool tc_supported(const FwdShape &sh, la_dtype dtype, int causal,
                  const void *q, const void *k, const void *v,
                  const void *out);

// Enqueues the tensor-core forward on `stream`.  `segment_chunks` = 0 picks
// the segment length automatically.  `status` is the device status word.
// `ws` (ws_bytes >= tc_workspace_bytes, 256-byte aligned) is the kernels'
// scratch; NULL makes the launch allocate it stream-ordered
// (cudaMallocAsync / cudaFreeAsync on `stream`).
// S_out / z_out (causal only, may be NULL, S_out 16-byte aligned): also
// write the final state [BH][d][d] / [BH][d] in fp32.
// gates (causal only, may be NULL): a device [BH][N] gate per token.
TcResult tc_forward(const void *q, const void *k, const void *v, void *out,
                    const FwdShape &sh, int causal, const DecayArgs &dk,
                    int segment_chunks, int *status, void *ws, size_t ws_bytes,
                    float *S_out, float *z_out, const float *gates,
                    cudaStream_t stream);

// CUDA-core (fp32 FMA) forward: any d in 1..LA_MAX_D, fp32 or bf16.
// S_out / z_out (causal only, may be NULL): the final state [BH][d][d] /
// [BH][d] in fp32.  gates (causal only, may be NULL): a device [BH][N]
// scalar gate per token, used instead of the per-head decay.
// `segment_chunks` (chunks of 32 tokens per segment; 0 = automatic) sets the
// sequence parallelism; more than one segment per head takes a
// stream-ordered workspace (tc_workspace_alloc).  `launches` receives the
// number of kernels enqueued.
TcResult launch_simt_forward(const void *q, const void *k, const void *v, void *out,
                             const FwdShape &sh, int causal, const DecayArgs &decay,
                             la_dtype dtype, float *S_out, float *z_out, const float *gates,
                             int segment_chunks, cudaStream_t stream, int *launches);

// Scratch bytes one tensor-core forward needs on a device with `sms` SMs.
size_t tc_workspace_bytes(const FwdShape &sh, int causal, bool decay,
                          int segment_chunks, int sms);

// Zeroes `bytes` (a multiple of 16, 16-byte aligned) of device memory with a
// small kernel on `stream`.  The kernels' workspaces (ticket counters and
// flags) are cleared this way rather than with cudaMemsetAsync: a memset can
// be queued on a copy engine behind unrelated copies of other streams (for
// example the input copies of la_forward_host), which would hold the kernel
// back until they finish.
cudaError_t tc_zero_words(void *p, size_t bytes, cudaStream_t stream);

// Stream-ordered workspace allocation of the forward launches (tensor-core
// kernels, and the CUDA-core kernels when they cut sequences into segments)
// (cudaMallocAsync), which the allocation-failure test hook can make fail.
cudaError_t tc_workspace_alloc(void **ws, size_t bytes, cudaStream_t stream);

// Test hooks, per calling thread, each consumed by the next launch that
// reads it (set through la_debug_inject_timeout / la_debug_fail_next_allocs):
// the next d = 128 causal launch bounds every wait by `wait_cycles` and
// segment `hold_segment` never publishes the state it holds (-1: all do);
// the next `n` workspace allocations fail.
void tc_debug_set_timeout(long long wait_cycles, int hold_segment);
bool tc_debug_take_timeout(long long *wait_cycles, int *hold_segment);
void tc_debug_fail_allocs(int n);

// Non-causal two-pass kernel (la_noncausal_tc.cu).
TcResult launch_noncausal_tc(const void *q, const void *k, const void *v,
                             void *out, const FwdShape &sh, int seg_chunks,
                             int *status, void *ws, size_t ws_bytes,
                             cudaStream_t stream);
size_t noncausal_tc_workspace_bytes(const FwdShape &sh, int seg_chunks, int sms);

// Chunkwise causal kernel (la_causal_tc.cu).
TcResult launch_causal_tc(const void *q, const void *k, const void *v,
                          void *out, const FwdShape &sh, const DecayArgs &dk,
                          int seg_chunks, int *status, void *ws, size_t ws_bytes,
                          float *S_out, float *z_out, const float *gates,
                          cudaStream_t stream);
size_t causal_tc_workspace_bytes(const FwdShape &sh, bool decay, int seg_chunks, int sms);

// d = 128 causal kernel, one CTA per (head, segment) over all value columns
// (la_causal_wide.cu); no gates.  launch_causal_wide takes a caller's
// workspace or allocates it stream-ordered; launch_causal_wide_fixed runs in
// a fixed device scratch of `cap` bytes (lengthening segments to fit) and
// allocates nothing.
TcResult launch_causal_wide(const void *q, const void *k, const void *v, void *out,
                            const FwdShape &sh, const DecayArgs &dk, int seg_chunks,
                            int *status, void *ws, size_t ws_bytes, float *S_out,
                            float *z_out, cudaStream_t stream);
TcResult launch_causal_wide_fixed(const void *q, const void *k, const void *v,
                                  void *out, const FwdShape &sh, const DecayArgs &dk,
                                  int *status, char *scratch, size_t cap,
                                  cudaStream_t stream);
size_t causal_wide_workspace_bytes(const FwdShape &sh, int seg_chunks, int sms);
// Automatic segment length (chunks) of the d = 128 kernel.
int wide_segment_chunks(long long heads, int nchunks, int sms);

}  // namespace la
