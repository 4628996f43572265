// The delta rule over whole sequences (DeltaNet; Gated DeltaNet with the
// forget gate), on CUDA cores in fp32.  The recurrence ("Story of Attention -
// Part 5: Linear Attention: Kernels, Decay, and Gating", section 7):
//   S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T,
//   o_t = S_t q_t,
// with one beta and one alpha per token and head (alpha = 1 without the
// gate), no feature map and no normaliser.  The state is stored S[a][c] (a
// key feature, c value column): the page's S transposed, as in the decode
// step, so (S k)[c] = sum_a S[a][c] k[a].
//
// The pages name a chunkwise form of this rule but do not give it; this is
// the recurrent form, token after token.  Its parallelism comes from the
// columns: column c of S_t depends only on column c of S_{t-1}, on k_t, and
// on v_t[c].  A CTA owns a block of W value columns of one head and walks
// the sequence with that block in registers.  A thread holds 4 columns x R
// key features.  The 8 threads that share a column group sit in one warp, so
// the two reductions per token (the prediction S k and the read S q) are
// warp shuffles, and a token needs no block-wide barrier.  The read of token
// t and the prediction for token t + 1 share one pass over the registers.
// Tokens are staged in shared memory 32 at a time, and the outputs leave
// through a staged tile.  Where rows are whole 16-byte vectors, the next
// chunk's q, k, v, beta and alpha are copied in with cp.async while the
// current chunk runs (double buffered, converted to fp32 in shared memory
// when their turn comes); otherwise each chunk is loaded when it is needed.
#include <cuda_bf16.h>

#include "la_internal.h"
#include "la_tc_host.h"

namespace la {
namespace {

constexpr int kT = 32;  // tokens per staged chunk

__device__ __forceinline__ float ld_in(const float *p) { return *p; }
__device__ __forceinline__ float ld_in(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
__device__ __forceinline__ void st_out(float *p, float x) { *p = x; }
__device__ __forceinline__ void st_out(__nv_bfloat16 *p, float x) {
    *p = __float2bfloat16_rn(x);
}

// Sum over the 8 row groups of a column group (lane bits 2-4).
__device__ __forceinline__ float sum_rows(float x) {
    x += __shfl_xor_sync(~0u, x, 4);
    x += __shfl_xor_sync(~0u, x, 8);
    x += __shfl_xor_sync(~0u, x, 16);
    return x;
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     (unsigned)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                     (unsigned)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}
__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

// Shared-memory floats of one CTA: k and q rows (8 row groups of R features,
// each padded to R + 4 so that the row groups' 16-byte reads fall in
// distinct banks), v and the outputs of this block's W columns, beta, alpha.
__host__ __device__ constexpr int delta_row(int R) { return 8 * (R + 4); }
__host__ __device__ constexpr int delta_smem_floats(int R, int W) {
    return 2 * kT * delta_row(R) + 2 * kT * W + 2 * kT;
}
// With asynchronous staging, two raw chunks (k, q rows of d elements, v of
// W columns, in the input type) and two raw beta / alpha rows follow.
__host__ __device__ constexpr size_t delta_raw_elems(int d, int W) {
    return (size_t)kT * (2 * d + W);
}

template <typename T, int R, bool kAsync>
__global__ void __launch_bounds__(256, 1)
delta_forward_kernel(const T *__restrict__ q, const T *__restrict__ k,
                     const T *__restrict__ v, T *__restrict__ out,
                     const float *__restrict__ beta, const float *__restrict__ alpha,
                     float *__restrict__ S, int N, int d, int W, int nsplit) {
    constexpr int RP = R + 4, DP = delta_row(R);
    extern __shared__ float4 smem4[];
    float *kb = reinterpret_cast<float *>(smem4);  // [kT][DP]
    float *qb = kb + kT * DP;                        // [kT][DP]
    float *vb = qb + kT * DP;                        // [kT][W]
    float *ob = vb + kT * W;                         // [kT][W]
    float *bb = ob + kT * W;                         // [kT]
    float *ab = bb + kT;                             // [kT]
    // asynchronous staging: raw chunk buffers b = 0, 1, then beta / alpha
    T *raw = reinterpret_cast<T *>(ab + kT);
    const size_t RAW = delta_raw_elems(d, W);
    float *fraw = reinterpret_cast<float *>(raw + 2 * RAW);  // [2][2][kT]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long bh = blockIdx.x / nsplit;
    const int c0 = (int)(blockIdx.x % nsplit) * W;
    const int cg = lane & 3, rg = lane >> 2;
    const int col = 16 * warp + 4 * cg;  // this thread's 4 columns in the block
    const int a0 = rg * R;               // its first key feature
    const size_t base = (size_t)bh * N * d;

    float s[R][4];
#pragma unroll
    for (int i = 0; i < R; ++i)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const int a = a0 + i, c = c0 + col + jj;
            s[i][jj] = (S && a < d && c < d) ? S[((size_t)bh * d + a) * d + c] : 0.f;
        }

    constexpr int VE = 16 / (int)sizeof(T);  // elements per 16-byte copy
    // issue the copies of chunk c into raw buffer b (asynchronous staging)
    auto stage = [&](int c, int b) {
        const int s0 = c * kT, m = min(kT, N - s0);
        T *kr = raw + b * RAW, *qr = kr + kT * d, *vr = qr + kT * d;
        const int nvr = d / VE, nvw = W / VE;
        for (int i = tid; i < m * nvr; i += blockDim.x) {
            const int t = i / nvr, e = (i - t * nvr) * VE;
            const size_t off = base + (size_t)(s0 + t) * d + e;
            cp_async16(kr + t * d + e, k + off);
            cp_async16(qr + t * d + e, q + off);
        }
        for (int i = tid; i < m * nvw; i += blockDim.x) {
            const int t = i / nvw, e = (i - t * nvw) * VE;
            if (c0 + e < d) cp_async16(vr + t * W + e, v + base + (size_t)(s0 + t) * d + c0 + e);
        }
        for (int i = tid; i < m; i += blockDim.x) {
            const size_t g = (size_t)bh * N + s0 + i;
            cp_async4(fraw + (2 * b) * kT + i, beta + g);
            if (alpha) cp_async4(fraw + (2 * b + 1) * kT + i, alpha + g);
        }
        cp_async_commit();
    };
    const int nchunk = (N + kT - 1) / kT;
    if (kAsync) stage(0, 0);

    for (int t0 = 0; t0 < N; t0 += kT) {
        const int n = min(kT, N - t0);
        if (kAsync) {
            // the next chunk's copies go out first; this chunk's have landed
            const int c = t0 / kT, b = c & 1;
            if (c + 1 < nchunk) {
                stage(c + 1, b ^ 1);
                cp_async_wait<1>();
            } else {
                cp_async_wait<0>();
            }
            __syncthreads();
            const T *kr = raw + b * RAW, *qr = kr + kT * d, *vr = qr + kT * d;
            for (int i = tid; i < n * 8 * R; i += blockDim.x) {
                const int t = i / (8 * R), a = i - t * 8 * R;
                const int slot = t * DP + (a / R) * RP + a % R;
                kb[slot] = a < d ? to_f(kr[t * d + a]) : 0.f;
                qb[slot] = a < d ? to_f(qr[t * d + a]) : 0.f;
            }
            for (int i = tid; i < n * W; i += blockDim.x) {
                const int t = i / W, cc = i - t * W;
                vb[i] = c0 + cc < d ? to_f(vr[t * W + cc]) : 0.f;
            }
            if (tid < n) {
                bb[tid] = fraw[(2 * b) * kT + tid];
                ab[tid] = alpha ? fraw[(2 * b + 1) * kT + tid] : 1.f;
            }
            __syncthreads();
        } else {
        // stage the chunk: k and q (every feature, zero past d), v of this
        // block's columns, beta and alpha
        for (int i = tid; i < kT * 8 * R; i += blockDim.x) {
            const int t = i / (8 * R), a = i - t * 8 * R;
            const int slot = t * DP + (a / R) * RP + a % R;
            float kv = 0.f, qv = 0.f;
            if (t < n && a < d) {
                const size_t off = base + (size_t)(t0 + t) * d + a;
                kv = ld_in(k + off);
                qv = ld_in(q + off);
            }
            kb[slot] = kv;
            qb[slot] = qv;
        }
        for (int i = tid; i < kT * W; i += blockDim.x) {
            const int t = i / W, c = c0 + (i - t * W);
            vb[i] = (t < n && c < d) ? ld_in(v + base + (size_t)(t0 + t) * d + c) : 0.f;
        }
        if (tid < kT) {
            const size_t g = (size_t)bh * N + t0 + tid;
            bb[tid] = tid < n ? beta[g] : 0.f;
            ab[tid] = tid < n && alpha ? alpha[g] : 1.f;
        }
        __syncthreads();
        }

        // the prediction S_{t-1} k_t for the chunk's first token
        float pred[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const float *kt = kb + rg * RP;
#pragma unroll
            for (int i4 = 0; i4 < R / 4; ++i4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(kt + 4 * i4);
                const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        pred[jj] = fmaf(s[4 * i4 + e][jj], kk[e], pred[jj]);
            }
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) pred[jj] = sum_rows(pred[jj]);
        }
        for (int t = 0; t < n; ++t) {
            const float b = bb[t], al = ab[t];
            const float4 v4 = *reinterpret_cast<const float4 *>(vb + t * W + col);
            const float u[4] = {b * (v4.x - al * pred[0]), b * (v4.y - al * pred[1]),
                                b * (v4.z - al * pred[2]), b * (v4.w - al * pred[3])};
            // S_t = alpha S_{t-1} + k_t u^T
            const float *kt = kb + t * DP + rg * RP;
#pragma unroll
            for (int i4 = 0; i4 < R / 4; ++i4) {
                const float4 k4 = *reinterpret_cast<const float4 *>(kt + 4 * i4);
                const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        s[4 * i4 + e][jj] = fmaf(kk[e], u[jj], al * s[4 * i4 + e][jj]);
            }
            // o_t = S_t q_t and the next token's prediction S_t k_{t+1}
            const float *qt = qb + t * DP + rg * RP;
            const float *kn = kb + (t + 1 < n ? t + 1 : t) * DP + rg * RP;
            float o[4] = {0.f, 0.f, 0.f, 0.f}, pn[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i4 = 0; i4 < R / 4; ++i4) {
                const float4 q4 = *reinterpret_cast<const float4 *>(qt + 4 * i4);
                const float4 k4 = *reinterpret_cast<const float4 *>(kn + 4 * i4);
                const float qq[4] = {q4.x, q4.y, q4.z, q4.w};
                const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        o[jj] = fmaf(s[4 * i4 + e][jj], qq[e], o[jj]);
                        pn[jj] = fmaf(s[4 * i4 + e][jj], kk[e], pn[jj]);
                    }
            }
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                o[jj] = sum_rows(o[jj]);
                pred[jj] = sum_rows(pn[jj]);
            }
            if (rg == 0)
                *reinterpret_cast<float4 *>(ob + t * W + col) = make_float4(o[0], o[1], o[2], o[3]);
        }
        __syncthreads();
        // the chunk's outputs (the next chunk's staging writes other buffers;
        // its token loop starts after the next barrier)
        for (int i = tid; i < n * W; i += blockDim.x) {
            const int t = i / W, c = c0 + (i - t * W);
            if (c < d) st_out(out + base + (size_t)(t0 + t) * d + c, ob[i]);
        }
    }

    if (S) {
#pragma unroll
        for (int i = 0; i < R; ++i)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                const int a = a0 + i, c = c0 + col + jj;
                if (a < d && c < d) S[((size_t)bh * d + a) * d + c] = s[i][jj];
            }
    }
}

template <typename T, int R>
cudaError_t launch_r(const void *q, const void *k, const void *v, void *out,
                     const float *beta, const float *alpha, float *S, long long BH,
                     int N, int d, int W, int nsplit, cudaStream_t stream) {
    // asynchronous staging needs whole 16-byte rows of q, k, v and room for
    // two raw chunks
    constexpr int VE = 16 / (int)sizeof(T);
    const size_t base_bytes = sizeof(float) * (size_t)delta_smem_floats(R, W);
    const size_t async_bytes = base_bytes + 2 * sizeof(T) * delta_raw_elems(d, W) +
                               sizeof(float) * 4 * kT;
    const bool async = d % VE == 0 && async_bytes <= 220 * 1024 &&
                       (reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                        reinterpret_cast<uintptr_t>(v)) % 16 == 0;
    const size_t smem = async ? async_bytes : base_bytes;
    auto kern = async ? delta_forward_kernel<T, R, true> : delta_forward_kernel<T, R, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(BH * nsplit), 2 * W, smem, stream>>>(
        static_cast<const T *>(q), static_cast<const T *>(k), static_cast<const T *>(v),
        static_cast<T *>(out), beta, alpha, S, N, d, W, nsplit);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const void *q, const void *k, const void *v, void *out,
                     const float *beta, const float *alpha, float *S, long long BH,
                     int N, int d, int W, int nsplit, cudaStream_t stream) {
    if (d <= 32) return launch_r<T, 4>(q, k, v, out, beta, alpha, S, BH, N, d, W, nsplit, stream);
    if (d <= 64) return launch_r<T, 8>(q, k, v, out, beta, alpha, S, BH, N, d, W, nsplit, stream);
    if (d <= 128)
        return launch_r<T, 16>(q, k, v, out, beta, alpha, S, BH, N, d, W, nsplit, stream);
    return launch_r<T, 32>(q, k, v, out, beta, alpha, S, BH, N, d, W, nsplit, stream);
}

}  // namespace

cudaError_t launch_delta_forward(const void *q, const void *k, const void *v, void *out,
                                 const float *beta, const float *alpha, float *S,
                                 long long BH, int N, int d, la_dtype dtype,
                                 cudaStream_t stream) {
    // column blocks of W = 16 .. 128 columns (one warp per 16): the fewest
    // blocks that give at least two CTAs per SM, else one warp per CTA
    int sms = 0;
    if (tchost::sm_count(&sms) != cudaSuccess || sms <= 0) sms = 1;
    const int cols = (d + 15) / 16 * 16;
    int W = 16, nsplit = cols / 16;
    for (int ns = 1; ns <= cols / 16; ++ns) {
        const int w = ((cols + ns - 1) / ns + 15) / 16 * 16;
        if (w > 128) continue;
        W = w;
        nsplit = (cols + w - 1) / w;
        if (BH * nsplit >= 2LL * sms) break;
    }
    if (BH * nsplit > 2147483647LL) return cudaErrorInvalidConfiguration;
    return dtype == LA_F32
               ? launch_t<float>(q, k, v, out, beta, alpha, S, BH, N, d, W, nsplit, stream)
               : launch_t<__nv_bfloat16>(q, k, v, out, beta, alpha, S, BH, N, d, W, nsplit,
                                         stream);
}

}  // namespace la
