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
TcResult tc_forward(const void *q, const void *k, const void *v, void *out,
                    const FwdShape &sh, int causal, const DecayArgs &dk,
                    int segment_chunks, int *status, cudaStream_t stream);

// Non-causal two-pass kernel (la_noncausal_tc.cu).
TcResult launch_noncausal_tc(const void *q, const void *k, const void *v,
                             void *out, const FwdShape &sh, int seg_chunks,
                             int *status, cudaStream_t stream);

// Chunkwise causal kernel (la_causal_tc.cu).
TcResult launch_causal_tc(const void *q, const void *k, const void *v,
                          void *out, const FwdShape &sh, const DecayArgs &dk,
                          int seg_chunks, int *status, cudaStream_t stream);

}  // namespace la
