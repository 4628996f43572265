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
                    int segment_chunks, int *status, cudaStream_t stream) {
    if (causal)
        return launch_causal_tc(q, k, v, out, sh, dk, segment_chunks, status,
                                stream);
    return launch_noncausal_tc(q, k, v, out, sh, segment_chunks, status, stream);
}

}  // namespace la
