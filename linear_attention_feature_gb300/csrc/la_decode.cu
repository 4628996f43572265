// Recurrent decode step: S <- g S + phi(k) v^T, z <- g z + phi(k),
// out = phi(q)^T S / phi(q)^T z  ("Linear Attention", running statistics and
// the O(d^2)-per-token inference cost; g the per-head decay of the
// forget-gate passage, 1 without decay).  g = 1 multiplies by one exactly, so
// the undecayed step is unchanged.  The retention variant ("Story of
// Attention - Part 5", section 4, recurrent form) uses the identity for phi
// and no denominator.  A device array of per-head gates (one per call: the
// data-dependent scalar gate alpha_t of this token) replaces the decay.
//
// The step is a pure stream over the fp32 d x d state (read once, written
// once): 2 * 4 * d^2 bytes per head against ~4 d^2 flops, so it is bound by
// HBM bandwidth.  One CTA owns one head.  In the vector kernel a thread owns
// 4 adjacent value columns c (one 128-bit load per state row) for a fixed
// subset of key-feature rows a; a warp therefore reads whole 512-byte rows
// (d = 128) perfectly coalesced.  All of a thread's rows are loaded before
// any is used so that its loads are in flight together.  The per-column
// partial sums of phi(q)^T S are reduced across row groups through shared
// memory; the denominator phi(q)^T z is reduced with warp shuffles.
#include <cuda_bf16.h>

#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;

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

// Shared prologue: phi(k), phi(q) into shared memory; z <- z + phi(k) and
// den = phi(q)^T z (after the update) reduced into *sden.
template <typename T>
__device__ __forceinline__ void decode_prologue(float *__restrict__ zh,
                                                const T *__restrict__ qh,
                                                const T *__restrict__ kh,
                                                int d, float g, bool use_phi,
                                                float *sk, float *sq,
                                                float *swarp, float *sden) {
    const int tid = threadIdx.x;
    float part = 0.f;
    for (int a = tid; a < d; a += kThreads) {
        float pk = fm(use_phi, ld_in(kh + a));
        float pq = fm(use_phi, ld_in(qh + a));
        sk[a] = pk;
        sq[a] = pq;
        float zn = fmaf(g, zh[a], pk);
        zh[a] = zn;
        part = fmaf(pq, zn, part);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
    if ((tid & 31) == 0) swarp[tid >> 5] = part;
    __syncthreads();
    if (tid == 0) {
        float s = 0.f;
        for (int w = 0; w < kThreads / 32; ++w) s += swarp[w];
        *sden = s;
    }
}

// d == D, D % 4 == 0, S 16-byte aligned.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
decode_vec_kernel(float *__restrict__ S, float *__restrict__ z,
                  const T *__restrict__ q, const T *__restrict__ k,
                  const T *__restrict__ v, T *__restrict__ out, DecayArgs dk,
                  int use_phi, int norm, const float *__restrict__ gates) {
    constexpr int NCG = D / 4;                 // column groups (float4 each)
    constexpr int NRG = kThreads / NCG;        // row groups
    constexpr int RPT = D / NRG;               // rows per thread
    constexpr int BATCH = RPT < 16 ? RPT : 16; // loads in flight per thread
    static_assert(NCG <= kThreads && kThreads % NCG == 0, "bad D");
    static_assert(D % NRG == 0 && RPT % BATCH == 0, "bad D");
    __shared__ float sk[D], sq[D];
    __shared__ float4 red[NRG][NCG];
    __shared__ float swarp[kThreads / 32], sden;

    const long long bh = blockIdx.x;
    const int tid = threadIdx.x;
    const int cg = tid % NCG, rg = tid / NCG;
    float4 *__restrict__ Sh = reinterpret_cast<float4 *>(S + (size_t)bh * D * D);
    const float g = gates ? gates[bh] : decay_of(dk, (int)bh);
    decode_prologue<T>(z + (size_t)bh * D, q + (size_t)bh * D,
                       k + (size_t)bh * D, D, g, use_phi != 0, sk, sq, swarp, &sden);
    const T *vh = v + (size_t)bh * D + 4 * cg;
    const float v0 = ld_in(vh), v1 = ld_in(vh + 1), v2 = ld_in(vh + 2),
                v3 = ld_in(vh + 3);
    __syncthreads();

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r0 = 0; r0 < RPT; r0 += BATCH) {
        float4 s[BATCH];
#pragma unroll
        for (int r = 0; r < BATCH; ++r)
            s[r] = __ldcs(Sh + (size_t)(rg + (r0 + r) * NRG) * NCG + cg);
#pragma unroll
        for (int r = 0; r < BATCH; ++r) {
            const int a = rg + (r0 + r) * NRG;
            const float pk = sk[a], pq = sq[a];
            s[r].x = fmaf(pk, v0, g * s[r].x);
            s[r].y = fmaf(pk, v1, g * s[r].y);
            s[r].z = fmaf(pk, v2, g * s[r].z);
            s[r].w = fmaf(pk, v3, g * s[r].w);
            __stcs(Sh + (size_t)a * NCG + cg, s[r]);
            acc.x = fmaf(pq, s[r].x, acc.x);
            acc.y = fmaf(pq, s[r].y, acc.y);
            acc.z = fmaf(pq, s[r].z, acc.z);
            acc.w = fmaf(pq, s[r].w, acc.w);
        }
    }
    red[rg][cg] = acc;
    __syncthreads();
    if (tid < NCG) {
        float4 t = red[0][tid];
#pragma unroll
        for (int r = 1; r < NRG; ++r) {
            float4 u = red[r][tid];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        const float inv = norm ? 1.f / sden : 1.f;
        T *o = out + (size_t)bh * D + 4 * tid;
        st_out(o, t.x * inv);
        st_out(o + 1, t.y * inv);
        st_out(o + 2, t.z * inv);
        st_out(o + 3, t.w * inv);
    }
}

// Any d (1..LA_MAX_D) and any alignment: a thread per value column, rows in
// sequence (each row read coalesced across the CTA).
template <typename T>
__global__ void __launch_bounds__(kThreads)
decode_generic_kernel(float *__restrict__ S, float *__restrict__ z,
                      const T *__restrict__ q, const T *__restrict__ k,
                      const T *__restrict__ v, T *__restrict__ out, int d,
                      DecayArgs dk, int use_phi, int norm,
                      const float *__restrict__ gates) {
    __shared__ float sk[LA_MAX_D], sq[LA_MAX_D];
    __shared__ float swarp[kThreads / 32], sden;
    const long long bh = blockIdx.x;
    float *Sh = S + (size_t)bh * d * d;
    const float g = gates ? gates[bh] : decay_of(dk, (int)bh);
    decode_prologue<T>(z + (size_t)bh * d, q + (size_t)bh * d,
                       k + (size_t)bh * d, d, g, use_phi != 0, sk, sq, swarp, &sden);
    __syncthreads();
    for (int c = threadIdx.x; c < d; c += kThreads) {
        const float vc = ld_in(v + (size_t)bh * d + c);
        float acc = 0.f;
        for (int a = 0; a < d; ++a) {
            float s = fmaf(sk[a], vc, g * Sh[(size_t)a * d + c]);
            Sh[(size_t)a * d + c] = s;
            acc = fmaf(sq[a], s, acc);
        }
        st_out(out + (size_t)bh * d + c, norm ? acc / sden : acc);
    }
}

// Delta rule ("Story of Attention - Part 5", section 7, Gated DeltaNet):
// S_t = alpha S_{t-1} + beta (v_t - alpha S_{t-1} k_t) k_t^T, o_t = S_t q_t,
// no feature map and no normaliser.  The state is stored S[a][c] (a key
// feature, c value column), so the page's S k_t is pred[c] = sum_a S[a][c]
// k[a] and the update is S[a][c] = alpha S[a][c] + beta k[a] (v[c] - alpha
// pred[c]).  The prediction needs the whole state before any of it changes:
// in the vector kernel each thread keeps its rows in registers across the
// two reductions, so the state is still read once and written once.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
delta_vec_kernel(float *__restrict__ S, const T *__restrict__ q,
                 const T *__restrict__ k, const T *__restrict__ v,
                 T *__restrict__ out, const float *__restrict__ beta,
                 const float *__restrict__ alpha) {
    constexpr int NCG = D / 4;           // column groups (float4 each)
    constexpr int NRG = kThreads / NCG;  // row groups
    constexpr int RPT = D / NRG;         // rows per thread
    static_assert(NCG <= kThreads && kThreads % NCG == 0 && D % NRG == 0, "bad D");
    __shared__ float sk[D], sq[D];
    __shared__ float4 red[NRG][NCG];
    __shared__ float4 spred[NCG];
    const long long bh = blockIdx.x;
    const int tid = threadIdx.x;
    const int cg = tid % NCG, rg = tid / NCG;
    float4 *__restrict__ Sh = reinterpret_cast<float4 *>(S + (size_t)bh * D * D);
    for (int a = tid; a < D; a += kThreads) {
        sk[a] = ld_in(k + (size_t)bh * D + a);
        sq[a] = ld_in(q + (size_t)bh * D + a);
    }
    const float b = beta[bh], g = alpha ? alpha[bh] : 1.f;
    const T *vh = v + (size_t)bh * D + 4 * cg;
    const float v0 = ld_in(vh), v1 = ld_in(vh + 1), v2 = ld_in(vh + 2), v3 = ld_in(vh + 3);
    float4 s[RPT];
#pragma unroll
    for (int r = 0; r < RPT; ++r) s[r] = __ldcs(Sh + (size_t)(rg + r * NRG) * NCG + cg);
    __syncthreads();
    // prediction S_{t-1} k for this thread's four columns, over its rows
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const float ka = sk[rg + r * NRG];
        acc.x = fmaf(ka, s[r].x, acc.x);
        acc.y = fmaf(ka, s[r].y, acc.y);
        acc.z = fmaf(ka, s[r].z, acc.z);
        acc.w = fmaf(ka, s[r].w, acc.w);
    }
    red[rg][cg] = acc;
    __syncthreads();
    if (tid < NCG) {
        float4 t = red[0][tid];
#pragma unroll
        for (int r = 1; r < NRG; ++r) {
            const float4 u = red[r][tid];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        spred[tid] = t;
    }
    __syncthreads();
    const float4 pr = spred[cg];
    const float d0 = v0 - g * pr.x, d1 = v1 - g * pr.y, d2 = v2 - g * pr.z,
                d3 = v3 - g * pr.w;
    // update, write back, and the read o = S_t q
    acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < RPT; ++r) {
        const int a = rg + r * NRG;
        const float kb = b * sk[a], qa = sq[a];
        s[r].x = fmaf(kb, d0, g * s[r].x);
        s[r].y = fmaf(kb, d1, g * s[r].y);
        s[r].z = fmaf(kb, d2, g * s[r].z);
        s[r].w = fmaf(kb, d3, g * s[r].w);
        __stcs(Sh + (size_t)a * NCG + cg, s[r]);
        acc.x = fmaf(qa, s[r].x, acc.x);
        acc.y = fmaf(qa, s[r].y, acc.y);
        acc.z = fmaf(qa, s[r].z, acc.z);
        acc.w = fmaf(qa, s[r].w, acc.w);
    }
    red[rg][cg] = acc;  // every read of red above finished before spred's barrier
    __syncthreads();
    if (tid < NCG) {
        float4 t = red[0][tid];
#pragma unroll
        for (int r = 1; r < NRG; ++r) {
            const float4 u = red[r][tid];
            t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
        }
        T *o = out + (size_t)bh * D + 4 * tid;
        st_out(o, t.x);
        st_out(o + 1, t.y);
        st_out(o + 2, t.z);
        st_out(o + 3, t.w);
    }
}

// Any d and alignment: a thread per value column; the state is read twice
// (prediction, then update).
template <typename T>
__global__ void __launch_bounds__(kThreads)
delta_generic_kernel(float *__restrict__ S, const T *__restrict__ q,
                     const T *__restrict__ k, const T *__restrict__ v,
                     T *__restrict__ out, const float *__restrict__ beta,
                     const float *__restrict__ alpha, int d) {
    __shared__ float sk[LA_MAX_D], sq[LA_MAX_D];
    const long long bh = blockIdx.x;
    float *Sh = S + (size_t)bh * d * d;
    for (int a = threadIdx.x; a < d; a += kThreads) {
        sk[a] = ld_in(k + (size_t)bh * d + a);
        sq[a] = ld_in(q + (size_t)bh * d + a);
    }
    __syncthreads();
    const float b = beta[bh], g = alpha ? alpha[bh] : 1.f;
    for (int c = threadIdx.x; c < d; c += kThreads) {
        float pred = 0.f;
        for (int a = 0; a < d; ++a) pred = fmaf(sk[a], Sh[(size_t)a * d + c], pred);
        const float dc = ld_in(v + (size_t)bh * d + c) - g * pred;
        float o = 0.f;
        for (int a = 0; a < d; ++a) {
            const float sn = fmaf(b * sk[a], dc, g * Sh[(size_t)a * d + c]);
            Sh[(size_t)a * d + c] = sn;
            o = fmaf(sq[a], sn, o);
        }
        st_out(out + (size_t)bh * d + c, o);
    }
}

template <typename T>
cudaError_t launch_delta_t(float *S, const void *q, const void *k, const void *v,
                           void *out, const float *beta, const float *alpha,
                           long long BH, int d, cudaStream_t stream) {
    const T *qq = static_cast<const T *>(q), *kk = static_cast<const T *>(k),
            *vv = static_cast<const T *>(v);
    T *oo = static_cast<T *>(out);
    const bool aligned = (reinterpret_cast<uintptr_t>(S) & 15u) == 0;
    dim3 grid((unsigned)BH);
    if (aligned && d == 128)
        delta_vec_kernel<T, 128><<<grid, kThreads, 0, stream>>>(S, qq, kk, vv, oo, beta, alpha);
    else if (aligned && d == 64)
        delta_vec_kernel<T, 64><<<grid, kThreads, 0, stream>>>(S, qq, kk, vv, oo, beta, alpha);
    else
        delta_generic_kernel<T><<<grid, kThreads, 0, stream>>>(S, qq, kk, vv, oo, beta, alpha, d);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(float *S, float *z, const void *q, const void *k,
                     const void *v, void *out, long long BH, int d,
                     const DecayArgs &dk, int phi, int norm, const float *gates,
                     cudaStream_t stream) {
    const T *qq = static_cast<const T *>(q), *kk = static_cast<const T *>(k),
            *vv = static_cast<const T *>(v);
    T *oo = static_cast<T *>(out);
    const bool aligned = (reinterpret_cast<uintptr_t>(S) & 15u) == 0;
    dim3 grid((unsigned)BH);
    if (aligned && d == 128)
        decode_vec_kernel<T, 128><<<grid, kThreads, 0, stream>>>(S, z, qq, kk, vv, oo, dk, phi, norm, gates);
    else if (aligned && d == 64)
        decode_vec_kernel<T, 64><<<grid, kThreads, 0, stream>>>(S, z, qq, kk, vv, oo, dk, phi, norm, gates);
    else if (aligned && d == 256)
        decode_vec_kernel<T, 256><<<grid, kThreads, 0, stream>>>(S, z, qq, kk, vv, oo, dk, phi, norm, gates);
    else
        decode_generic_kernel<T><<<grid, kThreads, 0, stream>>>(S, z, qq, kk, vv, oo, d, dk, phi, norm, gates);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_delta_step(float *S, const void *q, const void *k,
                              const void *v, void *out, const float *beta,
                              const float *alpha, long long BH, int d,
                              la_dtype dtype, cudaStream_t stream) {
    if (dtype == LA_F32)
        return launch_delta_t<float>(S, q, k, v, out, beta, alpha, BH, d, stream);
    return launch_delta_t<__nv_bfloat16>(S, q, k, v, out, beta, alpha, BH, d, stream);
}

cudaError_t launch_decode_step(float *S, float *z, const void *q,
                               const void *k, const void *v, void *out,
                               long long BH, int d, const DecayArgs &dk,
                               int phi, int norm, const float *gates,
                               la_dtype dtype, cudaStream_t stream) {
    if (dtype == LA_F32)
        return launch_t<float>(S, z, q, k, v, out, BH, d, dk, phi, norm, gates, stream);
    return launch_t<__nv_bfloat16>(S, z, q, k, v, out, BH, d, dk, phi, norm, gates, stream);
}

}  // namespace la
