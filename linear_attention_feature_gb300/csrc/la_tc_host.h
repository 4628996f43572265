// Host-side helpers for the tensor-core kernels: TMA tensor maps over the
// [B*H][N][d] bf16 sequences and per-device properties.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <utility>

namespace la {
namespace tchost {

// cuTensorMapEncodeTiled, fetched once through the runtime (no -lcuda).
inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn(cudaError_t *err) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static cudaError_t st = cudaSuccess;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        st = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled",
                                              reinterpret_cast<void **>(&fn),
                                              12000, cudaEnableDefault, &q);
        if (st == cudaSuccess && q != cudaDriverEntryPointSuccess)
            st = cudaErrorNotSupported;
    });
    *err = st;
    return fn;
}

// 3-D map over a contiguous bf16 tensor viewed as [BH][N][d] (d fastest),
// box = {64 features, rows tokens, 1 head}, 128-byte swizzle, zero fill out
// of bounds (rows past N read as 0; stores past N are dropped).
inline cudaError_t make_seq_map(CUtensorMap *map, const void *base, int BH,
                                int N, int d, int rows) {
    cudaError_t err;
    auto enc = encode_fn(&err);
    if (!enc) return err == cudaSuccess ? cudaErrorNotSupported : err;
    cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)N, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)N * d * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                     const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Number of SMs of the current device (cached per device).
inline cudaError_t sm_count(int *out) {
    static std::mutex mu;
    static int cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev]) {
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        cache[dev] = n;
    }
    *out = cache[dev];
    return cudaSuccess;
}

// Launches `kern` on `stream` with programmatic stream serialisation: its
// CTAs may start (barrier set-up, TMEM allocation, descriptor prefetch)
// while the kernel before it in the stream, the workspace clear, still runs.
// The kernel calls griddepcontrol.wait before it touches any global memory.
template <typename... P, typename... A>
inline cudaError_t launch_dependent(void (*kern)(P...), unsigned grid, unsigned block,
                                    size_t smem, cudaStream_t stream, A &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<A>(args)...);
}

// Chunks per sequence segment for the persistent tensor-core kernels.  A
// work item is one segment of one head (and value half), and the one-CTA-
// per-SM grid takes items in waves of `sms`.  The length chosen minimises
//   ceil(items / sms) * (segment length + overhead),
// with `overhead` the per-item cost (state publication, look-back) in chunk
// times; a head in one segment has none.  Longer segments win ties.
inline int wave_segment_chunks(long long heads, int nchunks, int sms, int overhead) {
    int best = nchunks;
    long long best_cost = -1;
    for (int len = nchunks; len >= 1; --len) {
        const long long nseg = (nchunks + len - 1) / len;
        const long long waves = (heads * nseg + sms - 1) / sms;
        const long long cost = waves * (len + (nseg > 1 ? overhead : 0));
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = len;
        }
    }
    return best;
}

}  // namespace tchost
}  // namespace la
