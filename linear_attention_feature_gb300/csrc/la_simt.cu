// CUDA-core (fp32 FMA, no tensor cores, no TF32) forward path.
//
// Serves fp32 inputs (where TF32 rounding would break a 1e-4 error budget)
// and bf16 inputs with a head dimension the tensor-core kernels do not take.
// Everything runs in fp32 with the chunkwise form of the recurrence
// ("Linear Attention", chunkwise parallel form: quadratic inside a chunk,
// state recurrence between chunks; "Story of Attention - Part 5", section 6
// block formulas), over chunks of T = 32 tokens:
//   A_ij  = (phi(q_i) . phi(k_j)) g^(i-j), j <= i            (intra-chunk)
//   num_i = sum_j A_ij v_j + g^(i+1) phi(q_i)^T S            (S: state before
//   den_i = sum_j A_ij     + g^(i+1) phi(q_i)^T z             the chunk)
//   S    <- g^n S + sum_t g^(n-1-t) phi(k_t) v_t^T,  z likewise
// With a data-dependent gate alpha_t per token (S_t = alpha_t S_{t-1} + ...)
// every power of g becomes the product of the gates it spans: g^(i-j) ->
// prod_{t=j+1..i} alpha_t, g^(i+1) -> prod_{t<=i} alpha_t, g^n -> the
// product over the chunk (products only, so a zero gate is exact).
//
// Sequence parallelism: each sequence is cut into segments of whole chunks
// and the work spread over (head, segment, block of 64 value columns) CTAs
// in up to three launches:
//   1. local   -- each segment but the last walks its chunks from a zero
//                 state and writes its local state L_s (and, per segment,
//                 the product G_s of its decay over all its tokens);
//   2. scan    -- per head and state element, in segment order:
//                 start_0 = 0, start_{s+1} = G_s start_s + L_s
//                 (the recurrence applied across segments), in place;
//   3. output  -- each segment walks its chunks again from start_s and
//                 writes its outputs (the last also the final state).
// The non-causal form reduces S = phi(K)^T V, z = phi(K)^T 1 the same way
// (local sums, then their sum in segment order) and reads them with every
// query.  A single segment needs neither of the first two launches (the
// non-causal form then needs no scan).  All sums run in a fixed order, so
// repeated calls give identical results.
#include <cuda_bf16.h>

#include <algorithm>

#include "la_internal.h"
#include "la_tc.h"
#include "la_tc_host.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kT = 32;    // tokens per chunk
constexpr int kCB = 64;   // value columns per CTA
constexpr int kLdA = 36;  // row stride of the score tile (floats)

enum Mode { LOCAL = 0, CAUSAL_OUT = 1, NONCAUSAL_OUT = 2 };

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

__device__ __forceinline__ void fma4(float4 &acc, float s, const float4 &x) {
    acc.x = fmaf(s, x.x, acc.x);
    acc.y = fmaf(s, x.y, acc.y);
    acc.z = fmaf(s, x.z, acc.z);
    acc.w = fmaf(s, x.w, acc.w);
}

__device__ __forceinline__ float dot4(const float4 &a, const float4 &b, float acc) {
    acc = fmaf(a.x, b.x, acc);
    acc = fmaf(a.y, b.y, acc);
    acc = fmaf(a.z, b.z, acc);
    return fmaf(a.w, b.w, acc);
}

struct SimtParams {
    int N, d, dp, ldf;   // dp: d rounded up to 4; ldf: row stride of phi tiles
    int ncb;             // blocks of kCB value columns
    int nseg, seg_chunks, grid_segs;  // segments; segments this launch covers
    int phi, norm;
    float *ws;           // [BH][nseg][d*d + d] segment states (NULL: none)
    float *wg;           // [BH][nseg] segment decay products
    float *S_out, *z_out;
    const float *gates;  // [BH][N] or NULL
};

// Shared-memory layout (floats).  The query tile, score tile and
// denominators come last: the local launch needs none of them.
struct SimtSmem {
    int S, z, K, V, gp, gt, gc, wv, Q, A, den, total;
    __host__ __device__ SimtSmem(int dp, int ldf, bool out) {
        S = 0;                      // [dp][kCB] state block
        z = S + dp * kCB;           // [dp]
        K = z + dp;                 // [kT][ldf] phi(k)
        V = K + kT * ldf;           // [kT][kCB]
        gp = V + kT * kCB;          // [36]: g^0 .. g^kT; [33] the chunk's decay
        gt = gp + 36;               // [kT][kT] decay from token j to i
        gc = gt + kT * kT;          // [kT] decay from the chunk start to i
        wv = gc + kT;               // [kT] weight of token t in the update
        Q = wv + kT;                // [kT][ldf] phi(q)
        A = Q + kT * ldf;           // [kT][kLdA] scores
        den = A + kT * kLdA;        // [kT]
        total = out ? den + kT : Q;
    }
};

// One CTA: head bh, segment seg, value columns [c0, c0 + 64) (see the file
// comment for the three modes).  256 threads; per chunk, four phases
// separated by barriers: tiles and decay tables; scores and denominators;
// numerators and outputs; state update.
template <typename T, int kMode>
__global__ void __launch_bounds__(kThreads, 4)
simt_chunk_kernel(const T *__restrict__ q, const T *__restrict__ k,
                  const T *__restrict__ v, T *__restrict__ out,
                  const SimtParams p, const DecayArgs decay) {
    extern __shared__ float4 smem4[];
    float *sm = reinterpret_cast<float *>(smem4);
    const SimtSmem L(p.dp, p.ldf, kMode != LOCAL);
    float *S = sm + L.S, *z = sm + L.z, *Ks = sm + L.K, *Vs = sm + L.V;
    float *gp = sm + L.gp, *gt = sm + L.gt, *gc = sm + L.gc, *wv = sm + L.wv;
    float *Qs = sm + L.Q, *A = sm + L.A, *den = sm + L.den;
    const float4 *S4 = reinterpret_cast<const float4 *>(S);
    const float4 *V4 = reinterpret_cast<const float4 *>(Vs);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const long long blk = blockIdx.x;
    const int cb = (int)(blk % p.ncb);
    const long long rest = blk / p.ncb;
    const int seg = (int)(rest % p.grid_segs);
    const long long bh = rest / p.grid_segs;
    const int d = p.d, dp = p.dp, ldf = p.ldf, d4 = p.dp / 4, ldf4 = p.ldf / 4;
    const int c0 = cb * kCB, cw = min(kCB, d - c0);
    const int nchunks = (p.N + kT - 1) / kT;
    const int ch0 = seg * p.seg_chunks, ch1 = min(ch0 + p.seg_chunks, nchunks);
    const size_t base = (size_t)bh * p.N * d;
    const size_t slot = (size_t)d * d + d;
    const bool gated = p.gates != nullptr, use_phi = p.phi != 0;

    // g^0 .. g^kT, each power by repeated multiplication in double
    if (tid == 0) {
        const double g = decay_of(decay, (int)(bh % decay.H));
        double x = 1.0;
        for (int i = 0; i <= kT; ++i, x *= g) gp[i] = (float)x;
    }
    // the state block: zero, or the segment's start state (causal) or the
    // whole sequence's state (non-causal)
    const float *st_in = nullptr;
    if (kMode == CAUSAL_OUT && p.ws) st_in = p.ws + ((size_t)bh * p.nseg + seg) * slot;
    if (kMode == NONCAUSAL_OUT) st_in = p.ws + (size_t)bh * p.nseg * slot;
    for (int i = tid; i < dp * kCB; i += kThreads) {
        const int a = i / kCB, c = i % kCB;
        S[i] = (st_in && a < d && c < cw) ? st_in[(size_t)a * d + c0 + c] : 0.f;
    }
    for (int a = tid; a < dp; a += kThreads) z[a] = (st_in && a < d) ? st_in[(size_t)d * d + a] : 0.f;
    double Gs = 1.0;  // LOCAL: decay over the segment (thread 0)
    __syncthreads();

    for (int ch = ch0; ch < ch1; ++ch) {
        const int t0 = ch * kT, n = min(kT, p.N - t0);
        // the state after this chunk is needed: to go on, or as the final state
        const bool upd = kMode == LOCAL ||
                         (kMode == CAUSAL_OUT &&
                          (ch + 1 < ch1 || (p.S_out && seg == p.nseg - 1)));
        // ---- 1. phi(q), phi(k), v tiles (zero past n and past d); decay tables
        for (int i = tid; i < kT * dp; i += kThreads) {
            const int t = i / dp, a = i - t * dp;
            float x = 0.f, y = 0.f;
            if (t < n && a < d) {
                const size_t off = base + (size_t)(t0 + t) * d + a;
                if (kMode != NONCAUSAL_OUT) x = fm(use_phi, ld_in(k + off));
                if (kMode != LOCAL) y = fm(use_phi, ld_in(q + off));
            }
            if (kMode != NONCAUSAL_OUT) Ks[t * ldf + a] = x;
            if (kMode != LOCAL) Qs[t * ldf + a] = y;
        }
        if (kMode != NONCAUSAL_OUT)
            for (int i = tid; i < kT * kCB; i += kThreads) {
                const int t = i / kCB, c = i % kCB;
                Vs[i] = (t < n && c < cw) ? ld_in(v + base + (size_t)(t0 + t) * d + c0 + c)
                                          : 0.f;
            }
        if (kMode != NONCAUSAL_OUT) {
            if (gated) {
                // lane t holds alpha of token t (1 past n)
                const float al = lane < n ? p.gates[(size_t)bh * p.N + t0 + lane] : 1.f;
                if (kMode == CAUSAL_OUT) {
                    // column j of the pairwise table: prefix products of the
                    // gates after token j (j = -1: from the chunk start)
                    for (int j = warp - 1; j < kT; j += kThreads / 32) {
                        float x = lane > j ? al : 1.f;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const float y = __shfl_up_sync(~0u, x, o);
                            if (lane >= o) x *= y;
                        }
                        if (j < 0)
                            gc[lane] = x;
                        else if (lane >= j)
                            gt[lane * kT + j] = x;
                    }
                }
                if (warp == 0) {
                    // suffix products: weight of token t in the update is the
                    // product of the gates after it; the chunk's decay is
                    // the product of all of them
                    float x = al;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float y = __shfl_down_sync(~0u, x, o);
                        if (lane + o < 32) x *= y;
                    }
                    const float after = __shfl_down_sync(~0u, x, 1);
                    wv[lane] = lane < n ? (lane == 31 ? 1.f : after) : 0.f;
                    if (lane == 0) gp[33] = x;
                }
            } else {
                if (tid < kT) wv[tid] = tid < n ? gp[n - 1 - tid] : 0.f;
                if (tid == kT) gp[33] = gp[n];
            }
        }
        __syncthreads();
        if (kMode == LOCAL && tid == 0) Gs *= (double)gp[33];

        if (kMode != LOCAL) {
            // ---- 2. scores (rows r, r+16; columns s, s+16) and denominators
            const int r = tid >> 4, s = tid & 15;
            const float4 *q0 = reinterpret_cast<const float4 *>(Qs + r * ldf);
            const float4 *q1 = reinterpret_cast<const float4 *>(Qs + (r + 16) * ldf);
            float rs0 = 0.f, rs1 = 0.f;  // row sums of the masked scores
            if (kMode == CAUSAL_OUT) {
                const float4 *k0 = reinterpret_cast<const float4 *>(Ks + s * ldf);
                const float4 *k1 = reinterpret_cast<const float4 *>(Ks + (s + 16) * ldf);
                // (r, s + 16) lies above the diagonal: no product
                float a00 = 0.f, a10 = 0.f, a11 = 0.f;
                for (int a4 = 0; a4 < d4; ++a4) {
                    const float4 x0 = q0[a4], x1 = q1[a4], y0 = k0[a4], y1 = k1[a4];
                    a00 = dot4(x0, y0, a00);
                    a10 = dot4(x1, y0, a10);
                    a11 = dot4(x1, y1, a11);
                }
                a00 = s <= r ? a00 * (gated ? gt[r * kT + s] : gp[r - s]) : 0.f;
                a10 = a10 * (gated ? gt[(r + 16) * kT + s] : gp[r + 16 - s]);
                a11 = s <= r ? a11 * (gated ? gt[(r + 16) * kT + s + 16] : gp[r - s]) : 0.f;
                A[r * kLdA + s] = a00;
                A[r * kLdA + s + 16] = 0.f;
                A[(r + 16) * kLdA + s] = a10;
                A[(r + 16) * kLdA + s + 16] = a11;
                rs0 = a00;
                rs1 = a10 + a11;
            }
            if (p.norm) {
                const float4 *z4 = reinterpret_cast<const float4 *>(z);
                float qz0 = 0.f, qz1 = 0.f;
                for (int a4 = s; a4 < d4; a4 += 16) {
                    const float4 zz = z4[a4];
                    qz0 = dot4(q0[a4], zz, qz0);
                    qz1 = dot4(q1[a4], zz, qz1);
                }
#pragma unroll
                for (int o = 1; o < 16; o <<= 1) {
                    rs0 += __shfl_xor_sync(~0u, rs0, o);
                    rs1 += __shfl_xor_sync(~0u, rs1, o);
                    qz0 += __shfl_xor_sync(~0u, qz0, o);
                    qz1 += __shfl_xor_sync(~0u, qz1, o);
                }
                if (s == 0) {
                    if (kMode == CAUSAL_OUT) {
                        den[r] = rs0 + (gated ? gc[r] : gp[r + 1]) * qz0;
                        den[r + 16] = rs1 + (gated ? gc[r + 16] : gp[r + 17]) * qz1;
                    } else {
                        den[r] = qz0;
                        den[r + 16] = qz1;
                    }
                }
            }
            __syncthreads();

            // ---- 3. numerators (rows r, r+16; columns 4 c4 .. 4 c4 + 3)
            const int c4 = tid & 15;
            if (4 * c4 < cw) {
                float4 n0 = make_float4(0.f, 0.f, 0.f, 0.f), n1 = n0, m0 = n0, m1 = n0;
                if (kMode == CAUSAL_OUT) {
                    const float4 *A0 = reinterpret_cast<const float4 *>(A + r * kLdA);
                    const float4 *A1 = reinterpret_cast<const float4 *>(A + (r + 16) * kLdA);
#pragma unroll 2
                    for (int j4 = 0; j4 < kT / 4; ++j4) {
                        const float4 x0 = A0[j4], x1 = A1[j4];
                        const float4 v0 = V4[(4 * j4) * (kCB / 4) + c4];
                        const float4 v1 = V4[(4 * j4 + 1) * (kCB / 4) + c4];
                        const float4 v2 = V4[(4 * j4 + 2) * (kCB / 4) + c4];
                        const float4 v3 = V4[(4 * j4 + 3) * (kCB / 4) + c4];
                        fma4(n0, x0.x, v0); fma4(n0, x0.y, v1); fma4(n0, x0.z, v2); fma4(n0, x0.w, v3);
                        fma4(n1, x1.x, v0); fma4(n1, x1.y, v1); fma4(n1, x1.z, v2); fma4(n1, x1.w, v3);
                    }
                }
#pragma unroll 2
                for (int a4 = 0; a4 < d4; ++a4) {
                    const float4 x0 = q0[a4], x1 = q1[a4];
                    const float4 s0 = S4[(4 * a4) * (kCB / 4) + c4];
                    const float4 s1 = S4[(4 * a4 + 1) * (kCB / 4) + c4];
                    const float4 s2 = S4[(4 * a4 + 2) * (kCB / 4) + c4];
                    const float4 s3 = S4[(4 * a4 + 3) * (kCB / 4) + c4];
                    fma4(m0, x0.x, s0); fma4(m0, x0.y, s1); fma4(m0, x0.z, s2); fma4(m0, x0.w, s3);
                    fma4(m1, x1.x, s0); fma4(m1, x1.y, s1); fma4(m1, x1.z, s2); fma4(m1, x1.w, s3);
                }
                const float g0 = kMode == CAUSAL_OUT ? (gated ? gc[r] : gp[r + 1]) : 1.f;
                const float g1 = kMode == CAUSAL_OUT ? (gated ? gc[r + 16] : gp[r + 17]) : 1.f;
                const float y0[4] = {fmaf(g0, m0.x, n0.x), fmaf(g0, m0.y, n0.y),
                                     fmaf(g0, m0.z, n0.z), fmaf(g0, m0.w, n0.w)};
                const float y1[4] = {fmaf(g1, m1.x, n1.x), fmaf(g1, m1.y, n1.y),
                                     fmaf(g1, m1.z, n1.z), fmaf(g1, m1.w, n1.w)};
                const float dn0 = p.norm ? den[r] : 1.f, dn1 = p.norm ? den[r + 16] : 1.f;
                const int cc = 4 * c4;
                for (int e = 0; e < 4 && cc + e < cw; ++e) {
                    if (r < n)
                        st_out(out + base + (size_t)(t0 + r) * d + c0 + cc + e,
                               p.norm ? y0[e] / dn0 : y0[e]);
                    if (r + 16 < n)
                        st_out(out + base + (size_t)(t0 + r + 16) * d + c0 + cc + e,
                               p.norm ? y1[e] / dn1 : y1[e]);
                }
            }
            __syncthreads();
        }

        // ---- 4. state update: S <- G S + sum_t w_t phi(k_t) v_t^T, z likewise
        if (upd) {
            const float G = gp[33];
            const float4 *K4 = reinterpret_cast<const float4 *>(Ks);
            float4 *Sw = reinterpret_cast<float4 *>(S);
            const int ntile = d4 * (kCB / 4);
            for (int tile = tid; tile < ntile; tile += kThreads) {
                const int a4 = tile / (kCB / 4), c4 = tile % (kCB / 4);
                if (4 * c4 >= cw) continue;
                float4 acc[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float4 x = Sw[(4 * a4 + u) * (kCB / 4) + c4];
                    acc[u] = make_float4(G * x.x, G * x.y, G * x.z, G * x.w);
                }
                for (int t = 0; t < n; ++t) {
                    const float w = wv[t];
                    const float4 kk = K4[t * ldf4 + a4];
                    const float4 vv = V4[t * (kCB / 4) + c4];
                    fma4(acc[0], w * kk.x, vv);
                    fma4(acc[1], w * kk.y, vv);
                    fma4(acc[2], w * kk.z, vv);
                    fma4(acc[3], w * kk.w, vv);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) Sw[(4 * a4 + u) * (kCB / 4) + c4] = acc[u];
            }
            for (int a = tid; a < dp; a += kThreads) {
                float s = G * z[a];
                for (int t = 0; t < n; ++t) s = fmaf(wv[t], Ks[t * ldf + a], s);
                z[a] = s;
            }
            __syncthreads();
        }
    }

    if (kMode == LOCAL) {
        // the segment's local state, its decay, into the segment's slot
        float *dst = p.ws + ((size_t)bh * p.nseg + seg) * slot;
        for (int i = tid; i < dp * kCB; i += kThreads) {
            const int a = i / kCB, c = i % kCB;
            if (a < d && c < cw) dst[(size_t)a * d + c0 + c] = S[i];
        }
        if (cb == 0) {
            for (int a = tid; a < d; a += kThreads) dst[(size_t)d * d + a] = z[a];
            if (tid == 0) p.wg[(size_t)bh * p.nseg + seg] = (float)Gs;
        }
    } else if (kMode == CAUSAL_OUT && p.S_out && seg == p.nseg - 1) {
        // the state after the last token, for a decode to continue from
        for (int i = tid; i < dp * kCB; i += kThreads) {
            const int a = i / kCB, c = i % kCB;
            if (a < d && c < cw) p.S_out[((size_t)bh * d + a) * d + c0 + c] = S[i];
        }
        if (cb == 0)
            for (int a = tid; a < d; a += kThreads) p.z_out[(size_t)bh * d + a] = z[a];
    }
}

// Per head and state element (d*d entries of S, then d of z), in segment
// order.  Causal: slot s <- start_s, with start_0 = 0 and start_{s+1} =
// G_s start_s + L_s (the last segment's slot holds no local state and only
// receives its start).  Non-causal: slot 0 <- the sum of all local sums.
__global__ void __launch_bounds__(kThreads)
simt_scan_kernel(float *__restrict__ ws, const float *__restrict__ wg, int nseg,
                 int d, int causal, int blocks_per_head) {
    const long long bh = blockIdx.x / blocks_per_head;
    const size_t slot = (size_t)d * d + d;
    const size_t e = (size_t)(blockIdx.x % blocks_per_head) * kThreads + threadIdx.x;
    if (e >= slot) return;
    float *x = ws + (size_t)bh * nseg * slot + e;
    float acc = 0.f;
    if (causal) {
        for (int s = 0; s < nseg; ++s) {
            const float l = s + 1 < nseg ? x[(size_t)s * slot] : 0.f;
            x[(size_t)s * slot] = acc;
            acc = fmaf(wg[(size_t)bh * nseg + s], acc, l);
        }
    } else {
        for (int s = 0; s < nseg; ++s) acc += x[(size_t)s * slot];
        x[0] = acc;
    }
}

template <typename T, int kMode>
cudaError_t launch_chunks(const void *q, const void *k, const void *v, void *out,
                          const SimtParams &p, const DecayArgs &decay, long long units,
                          cudaStream_t stream) {
    const size_t smem = sizeof(float) * (size_t)SimtSmem(p.dp, p.ldf, kMode != LOCAL).total;
    auto kern = simt_chunk_kernel<T, kMode>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)(units * p.grid_segs), kThreads, smem, stream>>>(
        static_cast<const T *>(q), static_cast<const T *>(k), static_cast<const T *>(v),
        static_cast<T *>(out), p, decay);
    return cudaGetLastError();
}

template <typename T>
TcResult launch_t(const void *q, const void *k, const void *v, void *out, const FwdShape &sh,
                  int causal, const DecayArgs &decay, float *S_out, float *z_out,
                  const float *gates, int segment_chunks, cudaStream_t stream,
                  int *launches) {
    SimtParams p{};
    p.N = sh.N;
    p.d = sh.d;
    p.dp = (sh.d + 3) / 4 * 4;
    // an odd number of 16-byte units per row keeps the column reads of the
    // score phase free of bank conflicts
    p.ldf = (p.dp / 4) % 2 ? p.dp : p.dp + 4;
    p.ncb = (sh.d + kCB - 1) / kCB;
    p.phi = sh.phi;
    p.norm = sh.norm;
    p.S_out = S_out;
    p.z_out = z_out;
    p.gates = gates;
    const long long BH = sh.BH(), units = BH * p.ncb;
    const int nchunks = (sh.N + kT - 1) / kT;
    // segments: as many as fill the GPU once with resident CTAs (one wave)
    int seg = segment_chunks;
    if (seg <= 0) {
        int sms = 0;
        if (tchost::sm_count(&sms) != cudaSuccess || sms <= 0) sms = 1;
        const size_t smem = sizeof(float) * (size_t)SimtSmem(p.dp, p.ldf, true).total + 1024;
        const long long per_sm = std::max<long long>(
            1, std::min<long long>(4, (long long)(232448 / smem)));
        const long long want = std::max<long long>(
            1, std::min<long long>(nchunks, sms * per_sm / std::max<long long>(units, 1)));
        seg = (int)((nchunks + want - 1) / want);
    }
    if (seg > nchunks) seg = nchunks;
    p.seg_chunks = seg;
    p.nseg = (nchunks + seg - 1) / seg;
    if ((double)units * p.nseg > 2147483647.0) {  // one segment per head then
        p.seg_chunks = nchunks;
        p.nseg = 1;
    }
    const size_t slot = (size_t)sh.d * sh.d + sh.d;
    const bool need_ws = !causal || p.nseg > 1;
    void *ws = nullptr;
    *launches = 0;
    if (need_ws) {
        const size_t states = sizeof(float) * slot * (size_t)BH * p.nseg;
        const size_t bytes = (states + 255) / 256 * 256 + sizeof(float) * (size_t)BH * p.nseg;
        cudaError_t e = tc_workspace_alloc(&ws, bytes, stream);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return {LA_ERR_NO_MEMORY, e, "la_forward: workspace allocation"};
        }
        p.ws = static_cast<float *>(ws);
        p.wg = reinterpret_cast<float *>(static_cast<char *>(ws) + (states + 255) / 256 * 256);
    }
    cudaError_t e = cudaSuccess;
    const int bph = (int)((slot + kThreads - 1) / kThreads);
    if (need_ws) {
        p.grid_segs = causal ? p.nseg - 1 : p.nseg;
        e = launch_chunks<T, LOCAL>(q, k, v, out, p, decay, units, stream);
        if (e == cudaSuccess) ++*launches;
        if (e == cudaSuccess && p.nseg > 1) {
            simt_scan_kernel<<<(unsigned)(BH * bph), kThreads, 0, stream>>>(
                p.ws, p.wg, p.nseg, sh.d, causal, bph);
            e = cudaGetLastError();
            if (e == cudaSuccess) ++*launches;
        }
    }
    if (e == cudaSuccess) {
        p.grid_segs = p.nseg;
        e = causal ? launch_chunks<T, CAUSAL_OUT>(q, k, v, out, p, decay, units, stream)
                   : launch_chunks<T, NONCAUSAL_OUT>(q, k, v, out, p, decay, units, stream);
        if (e == cudaSuccess) ++*launches;
    }
    if (ws) {
        const cudaError_t ef = cudaFreeAsync(ws, stream);
        if (e == cudaSuccess) e = ef;
    }
    if (e != cudaSuccess) return {LA_ERR_CUDA, e, "la_forward (CUDA-core kernels)"};
    return {LA_OK, cudaSuccess, nullptr};
}

}  // namespace

TcResult launch_simt_forward(const void *q, const void *k, const void *v, void *out,
                             const FwdShape &sh, int causal, const DecayArgs &decay,
                             la_dtype dtype, float *S_out, float *z_out, const float *gates,
                             int segment_chunks, cudaStream_t stream, int *launches) {
    if (!causal) {
        S_out = z_out = nullptr;
        gates = nullptr;
    }
    if (dtype == LA_F32)
        return launch_t<float>(q, k, v, out, sh, causal, decay, S_out, z_out, gates,
                               segment_chunks, stream, launches);
    return launch_t<__nv_bfloat16>(q, k, v, out, sh, causal, decay, S_out, z_out, gates,
                                   segment_chunks, stream, launches);
}

}  // namespace la
