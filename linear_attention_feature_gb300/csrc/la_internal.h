// Internal declarations shared by the translation units of liblinattn.so.
// Nothing here is part of the public ABI (include/linattn.h is).
#pragma once

#include <cuda_runtime.h>
#include <cstdint>

#include "linattn.h"

namespace la {

// Debug builds (-DLA_DEBUG) check the computed indices of the tensor-core
// kernels' global-memory accesses on the device.  A failed check records
// LA_ERR_INTERNAL and the source line in the device status word (the first
// failure wins; la_check_device_status reports it), and the guarded access
// is skipped.  Release builds compile the checks away: LA_DCHECK is `true`
// there and its condition is not evaluated.
#if defined(__CUDACC__) && defined(LA_DEBUG)
__device__ __forceinline__ bool dcheck_failed(int *status, int line) {
    if (atomicCAS(status, 0, (int)LA_ERR_INTERNAL) == 0) atomicExch(status + 1, line);
    return false;
}
#define LA_DCHECK(status, cond) ((cond) ? true : ::la::dcheck_failed((status), __LINE__))
#else
#define LA_DCHECK(status, cond) true
#endif

// Per-head decay, passed to kernels by value (kernel parameter space).
// has == 0 means g = 1 for every head.
struct DecayArgs {
    int has;
    int H;
    float g[LA_MAX_DECAY_HEADS];
};

__host__ __device__ inline float decay_of(const DecayArgs &dk, int bh) {
    return dk.has ? dk.g[bh % dk.H] : 1.0f;
}

// Common shape of a full-sequence call, with the method variant: phi = 1
// applies elu(x) + 1 to q and k (0: identity), norm = 1 divides by the
// normaliser phi(q)^T z (0: no denominator, as in retention).
struct FwdShape {
    int B, H, N, d;
    int phi = 1, norm = 1;
    long long BH() const { return (long long)B * H; }
};

// ---- delta-rule decode step (S only; beta, alpha device [BH], alpha may
// be NULL) ----
cudaError_t launch_delta_step(float *S, const void *q, const void *k,
                              const void *v, void *out, const float *beta,
                              const float *alpha, long long BH, int d,
                              la_dtype dtype, cudaStream_t stream);

// ---- delta rule over whole sequences (beta, alpha device [BH][N], alpha may
// be NULL; S device [BH][d][d] start and final state, or NULL for a zero
// start) ----
cudaError_t launch_delta_forward(const void *q, const void *k, const void *v, void *out,
                                 const float *beta, const float *alpha, float *S,
                                 long long BH, int N, int d, la_dtype dtype,
                                 cudaStream_t stream);

// ---- recurrent decode step ----
// phi / norm as in FwdShape; gates (may be NULL): a device [BH] gate per
// head for this step, used instead of the per-head decay.
cudaError_t launch_decode_step(float *S, float *z, const void *q,
                               const void *k, const void *v, void *out,
                               long long BH, int d, const DecayArgs &decay,
                               int phi, int norm, const float *gates,
                               la_dtype dtype, cudaStream_t stream);

// Address of the current device's two status words (kernels set word 0 to a
// non-zero la_status when a bounded wait gives up, and word 1 to where).
// Looked up once per device.
int *device_status_word(cudaError_t *err);

// Counts every kernel enqueued by the library (la_kernel_launch_count).
void note_launches(int n);

// Records the detail returned by la_last_error() on the calling thread.
void set_last_error(const char *msg);

// la_forward_ex with an optional caller-owned scratch for the tensor-core
// kernels (ws = NULL: they allocate it stream-ordered themselves).
// S_out / z_out (causal only, may be NULL): also write the final state.
// `variant` NULL: elu(x) + 1 with the normaliser.
// gates (causal only, may be NULL): a device [B][H][N] scalar gate per
// token, instead of `decay` (CUDA-core kernels).
la_status forward_with_workspace(const void *q, const void *k, const void *v,
                                 void *out, int B, int H, int N, int d,
                                 int causal, const float *decay, la_dtype dtype,
                                 int path, int segment_chunks, void *ws,
                                 size_t ws_bytes, float *S_out, float *z_out,
                                 const la_variant *variant, const float *gates,
                                 la_stream_t stream);

// The decode step behind la_decode_step(_ex/_variant/_gated): decay (host
// [H]) or gates (device [BH]), not both.
la_status decode_common(float *S, float *z, const void *q, const void *k,
                        const void *v, void *out, int B, int H, int d,
                        const float *decay, const float *gates, la_dtype dtype,
                        const la_variant *variant, la_stream_t stream);

// Scratch bytes forward_with_workspace needs (automatic path and segment
// length; 0 where the CUDA-core kernels run, which need none).
size_t forward_workspace_bytes(int B, int H, int N, int d, int causal,
                               bool decay, la_dtype dtype);

}  // namespace la
