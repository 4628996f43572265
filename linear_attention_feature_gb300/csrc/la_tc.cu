// Tensor-core forward kernels (placeholder until the tcgen05 kernels land).
#include "la_tc.h"

namespace la {

bool tc_supported(const FwdShape &, la_dtype) { return false; }

TcResult tc_forward(const void *, const void *, const void *, void *,
                    const FwdShape &, int, const DecayArgs &, int, int *,
                    cudaStream_t) {
    return {LA_ERR_UNSUPPORTED, cudaSuccess, "tensor-core path not built"};
}

}  // namespace la
