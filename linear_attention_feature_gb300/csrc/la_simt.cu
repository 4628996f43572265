// CUDA-core (fp32 FMA, no tensor cores, no TF32) forward path.
//
// Serves fp32 inputs (where TF32 rounding would break a 1e-4 error budget)
// and bf16 inputs with a head dimension the tensor-core kernels do not take.
// One CTA owns one (batch*head, block of 64 value columns) and walks the
// sequence in chunks of T = 32 tokens using the chunkwise form of the
// recurrence ("Linear Attention", chunkwise parallel form: quadratic inside a
// chunk, state recurrence between chunks; "Story of Attention - Part 5",
// section 6 block formulas), all in fp32:
//   A_ij  = (phi(q_i) . phi(k_j)) g^(i-j), j <= i            (intra-chunk)
//   num_i = sum_j A_ij v_j + g^(i+1) phi(q_i)^T S            (S: state before
//   den_i = sum_j A_ij     + g^(i+1) phi(q_i)^T z             the chunk)
//   S    <- g^n S + sum_t g^(n-1-t) phi(k_t) v_t^T,  z likewise
// With a data-dependent gate alpha_t per token (S_t = alpha_t S_{t-1} + ...)
// every power of g becomes the product of the gates it spans: g^(i-j) ->
// prod_{t=j+1..i} alpha_t, g^(i+1) -> prod_{t<=i} alpha_t, g^n -> the
// product over the chunk (a per-chunk table, so a zero gate is exact).
// The non-causal form first reduces S = phi(K)^T V and z = phi(K)^T 1 over
// the whole sequence, then reads them with every query.
#include <cuda_bf16.h>

#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kT = 32;   // tokens per chunk
constexpr int kCB = 64;  // value columns per CTA

__device__ __forceinline__ float ld_in(const float *p) { return *p; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
__device__ __forceinline__ void st_out(float *p, float x) { *p = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16 *p, float x) {
    *p = __float2bfloat16_rn(x);
}

// elu(x) + 1, alpha = 1; the identity when `use_phi` is false
__device__ __forceinline__ float fm(bool use_phi, float x) {
    return use_phi ? (x > 0.f ? x + 1.f : expf(x)) : x;
}

template <typename T, bool kCausal>
__global__ void __launch_bounds__(kThreads)
simt_forward_kernel(const T *__restrict__ q, const T *__restrict__ k,
                    const T *__restrict__ v, T *__restrict__ out, int N,
                    int d, DecayArgs decay, float *__restrict__ S_out,
                    float *__restrict__ z_out, int use_phi, int norm,
                    const float *__restrict__ gates) {
    extern __shared__ float smem[];
    const int cb = blockIdx.x;
    const long long bh = blockIdx.y;
    const int c0 = cb * kCB;
    const int cw = min(kCB, d - c0);
    float *S = smem;                  // [d][kCB]
    float *z = S + d * kCB;           // [d]
    float *pq = z + d;                // [kT][d]
    float *pk = pq + kT * d;          // [kT][d]
    float *pv = pk + kT * d;          // [kT][kCB]
    float *A = pv + kT * kCB;         // [kT][kT]
    float *den = A + kT * kT;         // [kT]
    float *gp = den + kT;             // [kT + 1]: g^0 .. g^kT
    float *gt = gp + kT + 1;          // [kT][kT]: prod_{t=j+1..i} alpha_t (gates)
    float *gc = gt + kT * kT;         // [kT]: prod_{t<=i} alpha_t (gates)

    const int tid = threadIdx.x;
    const size_t base = (size_t)bh * (size_t)N * (size_t)d;
    if (tid == 0) {
        double g = decay_of(decay, (int)bh), p = 1.0;
        for (int i = 0; i <= kT; ++i) { gp[i] = (float)p; p *= g; }
    }
    for (int i = tid; i < d * kCB; i += kThreads) S[i] = 0.f;
    for (int i = tid; i < d; i += kThreads) z[i] = 0.f;
    __syncthreads();

    if constexpr (!kCausal) {
        // pass 1: S = sum_j phi(k_j) v_j^T, z = sum_j phi(k_j)
        for (int t0 = 0; t0 < N; t0 += kT) {
            const int n = min(kT, N - t0);
            for (int i = tid; i < n * d; i += kThreads)
                pk[i] = fm(use_phi, ld_in(k + base + (size_t)t0 * d + i));
            for (int i = tid; i < n * kCB; i += kThreads) {
                int t = i / kCB, c = i % kCB;
                pv[i] = c < cw ? ld_in(v + base + (size_t)(t0 + t) * d + c0 + c)
                               : 0.f;
            }
            __syncthreads();
            for (int i = tid; i < d * kCB; i += kThreads) {
                int a = i / kCB, c = i % kCB;
                float s = S[i];
                for (int t = 0; t < n; ++t) s = fmaf(pk[t * d + a], pv[t * kCB + c], s);
                S[i] = s;
            }
            for (int a = tid; a < d; a += kThreads) {
                float s = z[a];
                for (int t = 0; t < n; ++t) s += pk[t * d + a];
                z[a] = s;
            }
            __syncthreads();
        }
        // pass 2: y_i = phi(q_i)^T S / phi(q_i)^T z
        for (int t0 = 0; t0 < N; t0 += kT) {
            const int n = min(kT, N - t0);
            for (int i = tid; i < n * d; i += kThreads)
                pq[i] = fm(use_phi, ld_in(q + base + (size_t)t0 * d + i));
            __syncthreads();
            for (int i = tid; i < n; i += kThreads) {
                float s = 0.f;
                for (int a = 0; a < d; ++a) s = fmaf(pq[i * d + a], z[a], s);
                den[i] = s;
            }
            __syncthreads();
            for (int i = tid; i < n * kCB; i += kThreads) {
                int t = i / kCB, c = i % kCB;
                if (c >= cw) continue;
                float s = 0.f;
                for (int a = 0; a < d; ++a) s = fmaf(pq[t * d + a], S[a * kCB + c], s);
                st_out(out + base + (size_t)(t0 + t) * d + c0 + c, norm ? s / den[t] : s);
            }
            __syncthreads();
        }
    } else {
    for (int t0 = 0; t0 < N; t0 += kT) {
        const int n = min(kT, N - t0);
        for (int i = tid; i < n * d; i += kThreads) {
            pq[i] = fm(use_phi, ld_in(q + base + (size_t)t0 * d + i));
            pk[i] = fm(use_phi, ld_in(k + base + (size_t)t0 * d + i));
        }
        for (int i = tid; i < n * kCB; i += kThreads) {
            int t = i / kCB, c = i % kCB;
            pv[i] = c < cw ? ld_in(v + base + (size_t)(t0 + t) * d + c0 + c) : 0.f;
        }
        if (gates) {
            // gate products of this chunk: thread j fills column j of the
            // table in order (gt[i][j] = gt[i-1][j] alpha_i), thread 0 the
            // prefix products
            const float *ga = gates + (size_t)bh * N + t0;
            if (tid < n) {
                float p = 1.f;
                gt[tid * kT + tid] = 1.f;
                for (int i = tid + 1; i < n; ++i) {
                    p *= ga[i];
                    gt[i * kT + tid] = p;
                }
            }
            if (tid == kThreads - 1) {
                float p = 1.f;
                for (int i = 0; i < n; ++i) {
                    p *= ga[i];
                    gc[i] = p;
                }
            }
        }
        __syncthreads();
        // intra-chunk masked, decayed scores
        for (int e = tid; e < kT * kT; e += kThreads) {
            int i = e / kT, j = e % kT;
            float a = 0.f;
            if (i < n && j <= i) {
                for (int f = 0; f < d; ++f) a = fmaf(pq[i * d + f], pk[j * d + f], a);
                a *= gates ? gt[i * kT + j] : gp[i - j];
            }
            A[e] = a;
        }
        __syncthreads();
        // denominators
        for (int i = tid; i < n; i += kThreads) {
            float s = 0.f, r = 0.f;
            for (int j = 0; j <= i; ++j) s += A[i * kT + j];
            for (int a = 0; a < d; ++a) r = fmaf(pq[i * d + a], z[a], r);
            den[i] = s + (gates ? gc[i] : gp[i + 1]) * r;
        }
        __syncthreads();
        // numerators and outputs
        for (int e = tid; e < n * kCB; e += kThreads) {
            int i = e / kCB, c = e % kCB;
            if (c >= cw) continue;
            float s = 0.f, r = 0.f;
            for (int j = 0; j <= i; ++j) s = fmaf(A[i * kT + j], pv[j * kCB + c], s);
            for (int a = 0; a < d; ++a) r = fmaf(pq[i * d + a], S[a * kCB + c], r);
            const float num = s + (gates ? gc[i] : gp[i + 1]) * r;
            st_out(out + base + (size_t)(t0 + i) * d + c0 + c, norm ? num / den[i] : num);
        }
        __syncthreads();
        // state update
        const float gall = gates ? gc[n - 1] : gp[n];
        for (int e = tid; e < d * kCB; e += kThreads) {
            int a = e / kCB, c = e % kCB;
            float s = gall * S[e];
            for (int t = 0; t < n; ++t) {
                const float w = gates ? gt[(n - 1) * kT + t] : gp[n - 1 - t];
                s = fmaf(w * pk[t * d + a], pv[t * kCB + c], s);
            }
            S[e] = s;
        }
        for (int a = tid; a < d; a += kThreads) {
            float s = gall * z[a];
            for (int t = 0; t < n; ++t)
                s = fmaf(gates ? gt[(n - 1) * kT + t] : gp[n - 1 - t], pk[t * d + a], s);
            z[a] = s;
        }
        __syncthreads();
    }
    // the state after the last token, for a decode to continue from
    if (S_out) {
        for (int e = tid; e < d * kCB; e += kThreads) {
            const int a = e / kCB, c = e % kCB;
            if (c < cw) S_out[((size_t)bh * d + a) * d + c0 + c] = S[e];
        }
        if (cb == 0)
            for (int a = tid; a < d; a += kThreads) z_out[(size_t)bh * d + a] = z[a];
    }
    }
}

template <typename T, bool kCausal>
cudaError_t launch_t(const void *q, const void *k, const void *v, void *out,
                     const FwdShape &sh, const DecayArgs &decay, float *S_out,
                     float *z_out, const float *gates, cudaStream_t stream) {
    const int d = sh.d;
    size_t smem_floats = (size_t)d * kCB + d + 2 * (size_t)kT * d +
                         (size_t)kT * kCB + kT * kT + kT + (kT + 1) +
                         (size_t)kT * kT + kT;
    size_t smem = smem_floats * sizeof(float);
    auto kern = simt_forward_kernel<T, kCausal>;
    cudaError_t e = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((d + kCB - 1) / kCB, (unsigned)sh.BH());
    kern<<<grid, kThreads, smem, stream>>>(
        static_cast<const T *>(q), static_cast<const T *>(k),
        static_cast<const T *>(v), static_cast<T *>(out), sh.N, d, decay, S_out,
        z_out, sh.phi, sh.norm, gates);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_forward(const void *q, const void *k, const void *v,
                                void *out, const FwdShape &sh, int causal,
                                const DecayArgs &decay, la_dtype dtype,
                                float *S_out, float *z_out, const float *gates,
                                cudaStream_t stream) {
    if (dtype == LA_F32)
        return causal ? launch_t<float, true>(q, k, v, out, sh, decay, S_out, z_out, gates, stream)
                      : launch_t<float, false>(q, k, v, out, sh, decay, nullptr, nullptr, nullptr, stream);
    return causal
               ? launch_t<__nv_bfloat16, true>(q, k, v, out, sh, decay, S_out, z_out, gates, stream)
               : launch_t<__nv_bfloat16, false>(q, k, v, out, sh, decay, nullptr, nullptr, nullptr, stream);
}

}  // namespace la
