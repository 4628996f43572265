// Non-causal linear attention on tcgen05 tensor cores (bf16 in, fp32
// accumulate): y_i = phi(q_i)^T S / phi(q_i)^T z with S = phi(K)^T V and
// z = phi(K)^T 1 over the whole sequence ("Story of Attention - Part 5",
// section 1a, matrix form phi(Q)[phi(K)^T V] / phi(Q)[phi(K)^T 1]; "Linear
// Attention", the two sums precomputed once per head and reused by every
// query).
//
// One persistent launch, two kinds of work item taken from one ticket
// counter:
//   pass 1 (head, segment, value half): S_seg | z_seg = phi(K)^T [V | 1] over
//     a run of 128-token chunks (tcgen05, N = 80, the ones column gives z),
//     written as an fp32 partial and counted in (an atomic per head).
//   pass 2 (head, chunk group, value half): waits (bounded) until all of its
//     head's partials are counted in, adds them in segment order -- so the
//     result does not depend on timing -- into the bf16 B operand, then per chunk
//     O | den = phi(Q) [S | z] (one N = 80 MMA per 16 features) into a
//     double-buffered TMEM accumulator, out = O / den, TMA store.
// Pass-1 tickets all precede pass-2 tickets and pass-1 items never wait, so
// every wait is on work held by a running CTA.
//
// Warp roles (448 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2-9 feature map (phi on packed bf16 pairs, in place), warps
// 10-13 state / output epilogue.
#include "la_tc.h"
#include "la_tc_common.cuh"
#include "la_tc_host.h"
#include "la_tc_ptx.cuh"

namespace la {
namespace noncausal_tc {

using namespace la::tc;
using namespace la::tcc;

constexpr int C = 128;
constexpr int DV = 64;
constexpr int NX = DV + 16;
constexpr int kWarpT = 2, kNumT = 8, kWarpE = 10;
constexpr int kThreads = (kWarpE + 4) * 32;  // 448
constexpr int kTThreads = kNumT * 32;
constexpr int BAR_T = 1, BAR_E = 2;
constexpr uint32_t TM_S = 0, TM_O0 = 96, TM_O1 = 176;  // 80 columns each
constexpr uint32_t TM_COLS = 256;

struct Params {
    int BH, N, nchunks, nhalf;
    int seg1, nseg1, items1;  // pass 1: chunks per segment, segments, items
    int grp2, ngrp2, items2;  // pass 2: chunks per group, groups, items
    float *part;              // [items1][STATE]
    int *cnt;                 // [BH * nhalf] partials counted in
    int phi, norm;            // elu(x) + 1 on q, k (else identity); divide by den
    int *ctrl;                // [0] ticket counter, [1] abort flag
    int *status;
    long long timeout;
};

template <int DK>
struct Layout {
    static constexpr int KB = DK / 64;
    static constexpr int STAGES = DK == 128 ? 3 : 4;
    static constexpr int TILE = DK * C * 2;   // K (pass 1) or Q (pass 2)
    static constexpr int VTILE = C * DV * 2;  // V half (pass 1) or O staging
    static constexpr int STAGE = TILE + VTILE;
    static constexpr int OFF_T = 0, OFF_V = TILE;
    static constexpr int OFF_SB = STAGES * STAGE;  // bf16 [S | z], MN-major
    static constexpr int SBLK = DK * 128;
    static constexpr int OFF_ONESX = OFF_SB + 2 * SBLK;  // ones column block
    static constexpr int ONESX = 16384;
    static constexpr int OFF_SMALL = OFF_ONESX + ONESX;
    static constexpr int STATE = DK * DV + DK;
};

struct Small {
    uint64_t full[4], empty[4], xf[4];
    uint64_t s_full, s_free, sb_ready, o_full[2], o_empty[2];
    uint64_t item_full[2], item_empty[2];
    uint64_t fin;  // every product of the CTA has completed (exit)
    int ring[2];
    uint32_t tmem_base;
};

struct Item {
    bool pass2;
    int bh, half, hh, c0, c1, seg;
};

__device__ __forceinline__ Item decode_item(int t, const Params &p) {
    Item it;
    it.pass2 = t >= p.items1;
    const int u0 = it.pass2 ? t - p.items1 : t;
    it.half = u0 % p.nhalf;
    const int u = u0 / p.nhalf;
    it.bh = u % p.BH;
    it.seg = u / p.BH;
    it.hh = it.bh * p.nhalf + it.half;
    const int per = it.pass2 ? p.grp2 : p.seg1;
    it.c0 = it.seg * per;
    it.c1 = min(it.c0 + per, p.nchunks);
    return it;
}

__device__ __forceinline__ int pop_item(Small &sm, int &tl, const Ctx &cx,
                                        int bar_id, int nthreads, bool leader) {
    const int r = tl & 1;
    settle_wait(&sm.item_full[r], (tl >> 1) & 1);
    const int t = ((volatile int *)sm.ring)[r];  // -1 once a wait gave up
    if (bar_id) named_bar_sync(bar_id, nthreads);
    if (leader) mbar_arrive(&sm.item_empty[r]);
    ++tl;
    return t;
}

template <int DK>
__device__ void producer(uint8_t *smem, Small &sm, const Params &p,
                         const Ctx &cx, const CUtensorMap *tq,
                         const CUtensorMap *tk, const CUtensorMap *tv) {
    using L = Layout<DK>;
    const uint64_t pol = policy_evict_first();
    const int total = p.items1 + p.items2;
    int j = 0, tl = 0;
    bool stop = false;  // a wait gave up: no further loads
    for (;;) {
        int t = atomicAdd(p.ctrl, 1);
        if (t >= total || stop || *cx.abort) t = -1;
        const int r = tl & 1;
        settle_wait(&sm.item_empty[r], ((tl >> 1) & 1) ^ 1);
        ((volatile int *)sm.ring)[r] = t;
        mbar_arrive(&sm.item_full[r]);
        ++tl;
        if (t < 0) break;
        const Item it = decode_item(t, p);
        for (int c = it.c0; c < it.c1; ++c, ++j) {
            const int st = j % L::STAGES;
            const uint32_t par = ((j / L::STAGES) & 1) ^ 1;
            if (!wait_bar(&sm.empty[st], par, cx)) {
                stop = true;
                break;
            }
            // one arming per phase: the slot's previous load has landed
            if (j >= L::STAGES) settle_wait(&sm.full[st], par);
            uint8_t *base = smem + st * L::STAGE;
            if (it.pass2) {
                mbar_arrive_expect_tx(&sm.full[st], L::TILE);
                for (int kb = 0; kb < L::KB; ++kb)
                    tma_load_3d(base + L::OFF_T + kb * 16384, tq, &sm.full[st],
                                64 * kb, c * C, it.bh, pol);
            } else {
                mbar_arrive_expect_tx(&sm.full[st], L::TILE + L::VTILE);
                for (int kb = 0; kb < L::KB; ++kb)
                    tma_load_3d(base + L::OFF_T + kb * 16384, tk, &sm.full[st],
                                64 * kb, c * C, it.bh, pol);
                tma_load_3d(base + L::OFF_V, tv, &sm.full[st], 64 * it.half,
                            c * C, it.bh, pol);
            }
        }
    }
    // the last load of each slot has landed before the CTA may exit
    for (int x = j - L::STAGES; x < j; ++x)
        if (x >= 0) settle_wait(&sm.full[x % L::STAGES], (x / L::STAGES) & 1);
}

template <int DK>
__device__ void mma_issuer(uint8_t *smem, Small &sm, const Params &p,
                           const Ctx &cx, uint32_t tmem) {
    using L = Layout<DK>;
    constexpr uint32_t idQS = idesc_bf16(128, NX, 0, 1);  // phi(Q) [S | z]
    constexpr uint32_t idSU = idesc_bf16(128, NX, 1, 1);  // phi(K)^T [V | 1]
    constexpr uint32_t lboA = DK == 128 ? 16384 : 0;      // d=64: rows alias
    const uint32_t sb = smem_u32(smem + L::OFF_SB);
    const uint32_t onesx = smem_u32(smem + L::OFF_ONESX);
    int j = 0, n1 = 0, n2 = 0, nb = 0, tl = 0;
    for (;;) {
        const int t = pop_item(sm, tl, cx, 0, 0, true);
        if (t < 0) break;
        const Item it = decode_item(t, p);
        if (!it.pass2) {
            wait_bar(&sm.s_free, (n1 & 1) ^ 1, cx);
            tc_fence_after();
            for (int c = it.c0; c < it.c1; ++c, ++j) {
                const int st = j % L::STAGES;
                wait_bar(&sm.xf[st], (j / L::STAGES) & 1, cx);
                tc_fence_after();
                const uint32_t kb = smem_u32(smem + st * L::STAGE + L::OFF_T);
                const uint32_t vb = smem_u32(smem + st * L::STAGE + L::OFF_V);
                for (int ks = 0; ks < C / 16; ++ks)
                    mma_ss(tmem + TM_S, sdesc_sw128(kb + ks * 2048, lboA, 1024),
                           sdesc_sw128(vb + ks * 2048, onesx - vb, 1024), idSU,
                           (c > it.c0 || ks > 0) ? 1u : 0u);
                mma_commit(&sm.empty[st]);
            }
            mma_commit(&sm.s_full);
            ++n1;
        } else {
            wait_bar(&sm.sb_ready, n2 & 1, cx);
            ++n2;
            for (int c = it.c0; c < it.c1; ++c, ++j, ++nb) {
                const int st = j % L::STAGES;
                const int ob = nb & 1;
                wait_bar(&sm.xf[st], (j / L::STAGES) & 1, cx);
                wait_bar(&sm.o_empty[ob], ((nb >> 1) & 1) ^ 1, cx);
                tc_fence_after();
                const uint32_t qb = smem_u32(smem + st * L::STAGE + L::OFF_T);
                for (int ks = 0; ks < DK / 16; ++ks)
                    mma_ss(tmem + (ob ? TM_O1 : TM_O0),
                           sdesc_sw128(qb + kmajor_off(ks, 16384), 16, 1024),
                           sdesc_sw128(sb + ks * 2048, L::SBLK, 1024), idQS,
                           ks > 0 ? 1u : 0u);
                mma_commit(&sm.o_full[ob]);
                mma_commit(&sm.empty[st]);
            }
        }
    }
    // every product has completed before TMEM is released
    mma_commit(&sm.fin);
    settle_wait(&sm.fin, 0);
}

// phi over this thread's half of one row of a [128][DK] swizzled tile, in
// place; rows past the sequence end become 0 when `zero` is set.
template <int DK>
__device__ __forceinline__ void transform_row(uint8_t *tile, int row, int part,
                                              bool zero, bool phi) {
    constexpr int NCH = DK / 16;
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
        const int cc = part * NCH + i;
        const uint32_t off = (cc >> 3) * 16384 + sw128_offset(row, (cc & 7) * 8);
        const uint4 x = *reinterpret_cast<const uint4 *>(tile + off);
        uint4 y = phi ? make_uint4(phi2(x.x), phi2(x.y), phi2(x.z), phi2(x.w)) : x;
        if (zero) y = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(tile + off) = y;
    }
}

template <int DK>
__device__ void transform(uint8_t *smem, Small &sm, const Params &p,
                          const Ctx &cx) {
    using L = Layout<DK>;
    const int et = threadIdx.x - kWarpT * 32;
    const int row = et & 127, part = et >> 7;
    int j = 0, tl = 0;
    for (;;) {
        const int t = pop_item(sm, tl, cx, BAR_T, kTThreads, et == 0);
        if (t < 0) break;
        const Item it = decode_item(t, p);
        for (int c = it.c0; c < it.c1; ++c, ++j) {
            const int st = j % L::STAGES;
            wait_bar(&sm.full[st], (j / L::STAGES) & 1, cx);
            // phi(K) rows past the end must be 0 (they would add keys);
            // phi(Q) rows past the end produce outputs that are not stored
            transform_row<DK>(smem + st * L::STAGE + L::OFF_T, row, part,
                              !it.pass2 && c * C + row >= p.N, p.phi);
            fence_async_shared();
            named_bar_sync(BAR_T, kTThreads);
            if (et == 0) mbar_arrive(&sm.xf[st]);
        }
    }
}

template <int DK>
__device__ void epilogue(uint8_t *smem, Small &sm, const Params &p,
                         const Ctx &cx, uint32_t tmem, const CUtensorMap *to) {
    using L = Layout<DK>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;
    const int row = q * 32 + lane;  // TMEM lane: S row a (pass 1) / query i
    const int et = threadIdx.x - kWarpE * 32;
    const bool act = row < DK;      // warp-uniform
    const uint32_t lb = tmem + ((uint32_t)(q * 32) << 16);
    uint8_t *sb = smem + L::OFF_SB;
    int j = 0, n1 = 0, nb = 0, tl = 0, pend = -1;
    for (;;) {
        const int t = pop_item(sm, tl, cx, BAR_E, 128, et == 0);
        if (t < 0) break;
        const Item it = decode_item(t, p);
        if (!it.pass2) {
            for (int c = it.c0; c < it.c1; ++c, ++j) {
                const int st = j % L::STAGES;
                wait_bar(&sm.full[st], (j / L::STAGES) & 1, cx);
                if (et == 0) mbar_arrive(&sm.empty[st]);
            }
            wait_bar(&sm.s_full, n1 & 1, cx);
            ++n1;
            tc_fence_after();
            float *dst = p.part + (size_t)t * L::STATE;
            if (act && LA_DCHECK(p.status, t >= 0 && t < p.items1 && row < DK)) {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t v[32];
                    tmem_ld32(lb + TM_S + 32 * h, v);
                    tmem_wait_ld();
                    reg_fence(v);
                    float4 *d4 = reinterpret_cast<float4 *>(dst + row * DV + 32 * h);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        d4[e] = make_float4(u2f(v[4 * e]), u2f(v[4 * e + 1]),
                                            u2f(v[4 * e + 2]), u2f(v[4 * e + 3]));
                }
                uint32_t zr = tmem_ld1(lb + TM_S + DV);
                tmem_wait_ld();
                reg_fence(zr);
                dst[DK * DV + row] = u2f(zr);
            }
            tc_fence_before();
            __threadfence();
            named_bar_sync(BAR_E, 128);
            if (et == 0) {
                mbar_arrive(&sm.s_free);
                atomicAdd(p.cnt + it.hh, 1);  // after the fence: the partial is visible
            }
            continue;
        }
        // pass 2: the head's [S | z] = sum of its partials in segment order,
        // staged in bf16.  For d = 64 two threads share a row (32 columns
        // each); for d = 128 each thread takes a row, both halves.
        if (warp == kWarpE) poll_flag_at_least(p.cnt + it.hh, p.nseg1, p.nseg1, cx);
        named_bar_sync(BAR_E, 128);
        {
            constexpr int NH = DK == 64 ? 1 : 2;
            const int a = DK == 64 ? (et & 63) : et;
            const int h0 = DK == 64 ? (et >> 6) : 0;
#pragma unroll 1
            for (int hh = 0; hh < NH; ++hh) {
                const int h = h0 + hh;
                const bool zh = h == 0;
                float acc[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) acc[e] = 0.f;
                float accz = 0.f;
#pragma unroll 2
                for (int s2 = 0; s2 < p.nseg1; ++s2) {
                    const int pi = (s2 * p.BH + it.bh) * p.nhalf + it.half;
                    if (!LA_DCHECK(p.status, pi >= 0 && pi < p.items1 && a < DK)) continue;
                    const float *src = p.part + (size_t)pi * L::STATE;
                    const float4 *s4 = reinterpret_cast<const float4 *>(src + a * DV + 32 * h);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float4 u = __ldcg(s4 + e);
                        acc[4 * e] += u.x;
                        acc[4 * e + 1] += u.y;
                        acc[4 * e + 2] += u.z;
                        acc[4 * e + 3] += u.w;
                    }
                    if (zh) accz += __ldcg(src + DK * DV + a);
                }
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    *reinterpret_cast<uint4 *>(sb + sw128_offset(a, 32 * h + ch * 8)) =
                        make_uint4(pack_bf16x2(acc[8 * ch], acc[8 * ch + 1]),
                                   pack_bf16x2(acc[8 * ch + 2], acc[8 * ch + 3]),
                                   pack_bf16x2(acc[8 * ch + 4], acc[8 * ch + 5]),
                                   pack_bf16x2(acc[8 * ch + 6], acc[8 * ch + 7]));
                if (zh)
                    *reinterpret_cast<__nv_bfloat16 *>(sb + L::SBLK + sw128_offset(a, 0)) =
                        __float2bfloat16_rn(accz);
            }
        }
        fence_async_shared();
        named_bar_sync(BAR_E, 128);
        if (et == 0) mbar_arrive(&sm.sb_ready);
        for (int c = it.c0; c < it.c1; ++c, ++j, ++nb) {
            const int st = j % L::STAGES;
            const int ob = nb & 1;
            const uint32_t tob = ob ? TM_O1 : TM_O0;
            wait_bar(&sm.o_full[ob], (nb >> 1) & 1, cx);
            tc_fence_after();
            uint32_t dreg = tmem_ld1(lb + tob + DV);
            uint32_t packed[32];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t o[32];
                tmem_ld32(lb + tob + 32 * h, o);
                tmem_wait_ld();
                reg_fence(o);
                reg_fence(dreg);
                const float inv = p.norm ? 1.f / u2f(dreg) : 1.f;
#pragma unroll
                for (int e = 0; e < 32; e += 2)
                    packed[16 * h + (e >> 1)] =
                        pack_bf16x2(u2f(o[e]) * inv, u2f(o[e + 1]) * inv);
            }
            tc_fence_before();
            mbar_arrive(&sm.o_empty[ob]);  // 128 arrivals: this row is read
            uint8_t *stage_o = smem + st * L::STAGE + L::OFF_V;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
                *reinterpret_cast<uint4 *>(stage_o + sw128_offset(row, ch * 8)) =
                    make_uint4(packed[4 * ch], packed[4 * ch + 1], packed[4 * ch + 2],
                               packed[4 * ch + 3]);
            fence_async_shared();
            named_bar_sync(BAR_E, 128);
            if (et == 0) {
                tma_store_3d(to, stage_o, 64 * it.half, c * C, it.bh);
                tma_store_commit();
                // release the previous chunk's stage once its store has
                // read it (one store stays in flight)
                if (pend >= 0) {
                    tma_store_wait_read<1>();
                    mbar_arrive(&sm.empty[pend]);
                }
                pend = st;
            }
        }
        if (et == 0 && pend >= 0) {  // the item's last store
            tma_store_wait_read<0>();
            mbar_arrive(&sm.empty[pend]);
            pend = -1;
        }
    }
    if (et == 0) tma_store_wait_all<0>();
}

template <int DK>
__global__ void __launch_bounds__(kThreads, 1)
noncausal_kernel(const __grid_constant__ CUtensorMap tq,
                 const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv,
                 const __grid_constant__ CUtensorMap to, const Params p) {
    using L = Layout<DK>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small &sm = *reinterpret_cast<Small *>(smem + L::OFF_SMALL);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Ctx cx{reinterpret_cast<volatile int *>(p.ctrl + 1), p.status,
                 p.timeout};
    if (threadIdx.x == 0) {
        for (int s = 0; s < L::STAGES; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 2);
            mbar_init(&sm.xf[s], 1);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.s_free, 1);
        mbar_init(&sm.sb_ready, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.o_full[b], 1);
            mbar_init(&sm.o_empty[b], 128);
            mbar_init(&sm.item_full[b], 1);
            mbar_init(&sm.item_empty[b], 3);  // MMA, transform, epilogue
        }
        mbar_init(&sm.fin, 1);
        fence_mbar_init();
    }
    // ones column of [V | 1]; the z block of [S | z] outside column 0 is zero
    for (int i = threadIdx.x; i < L::ONESX / 16; i += kThreads)
        reinterpret_cast<uint4 *>(smem + L::OFF_ONESX)[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < L::SBLK / 16; i += kThreads)
        reinterpret_cast<uint4 *>(smem + L::OFF_SB + L::SBLK)[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    if (threadIdx.x < C)
        *reinterpret_cast<uint16_t *>(smem + L::OFF_ONESX + sw128_offset(threadIdx.x, 0)) =
            (uint16_t)(kBf16One2 & 0xFFFFu);
    fence_async_shared();
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, TM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
        tma_prefetch_desc(&to);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the workspace clear before this kernel has completed (dependent launch)
    grid_dep_wait();
    const uint32_t tmem = sm.tmem_base;
    if (warp == 0) {
        if (lane == 0) producer<DK>(smem, sm, p, cx, &tq, &tk, &tv);
    } else if (warp == 1) {
        if (lane == 0) mma_issuer<DK>(smem, sm, p, cx, tmem);
    } else if (warp < kWarpE) {
        transform<DK>(smem, sm, p, cx);
    } else {
        epilogue<DK>(smem, sm, p, cx, tmem, &to);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TM_COLS);
}

template <int DK>
constexpr size_t smem_bytes() {
    return (size_t)Layout<DK>::OFF_SMALL + sizeof(Small) + 1024;
}
static_assert(smem_bytes<128>() <= 232448, "shared memory budget");
static_assert(smem_bytes<64>() <= 232448, "shared memory budget");

}  // namespace noncausal_tc

namespace {

inline size_t nc_align(size_t x) { return (x + 255) / 256 * 256; }

// Work decomposition and workspace layout of one non-causal launch.
struct NcPlan {
    int per, nseg, nchunks, nhalf;
    long long heads, items;
    size_t off_cnt, off_part, total;
};

template <int DK>
NcPlan plan_noncausal(const FwdShape &sh, int seg_chunks, int sms) {
    using namespace noncausal_tc;
    using L = Layout<DK>;
    NcPlan pl{};
    pl.nchunks = (sh.N + C - 1) / C;
    pl.nhalf = DK / DV;
    pl.heads = sh.BH() * pl.nhalf;
    // segment length by the wave rule (per-item overhead about three chunk
    // times, measured)
    pl.per = seg_chunks > 0 ? seg_chunks
                            : tchost::wave_segment_chunks(pl.heads, pl.nchunks, sms, 3);
    pl.nseg = (pl.nchunks + pl.per - 1) / pl.per;
    pl.items = pl.heads * pl.nseg;
    // workspace: control words, per-head counts (zeroed), partial states
    pl.off_cnt = 256;
    pl.off_part = nc_align(pl.off_cnt + sizeof(int) * (size_t)pl.heads);
    pl.total = pl.off_part + sizeof(float) * L::STATE * (size_t)pl.items;
    return pl;
}

template <int DK>
TcResult launch_noncausal_t(const void *q, const void *k, const void *v,
                            void *out, const FwdShape &sh, int seg_chunks,
                            int *status, void *ws_in, size_t ws_bytes,
                            cudaStream_t stream) {
    using namespace noncausal_tc;
    const int BH = (int)sh.BH(), N = sh.N;
    CUtensorMap tq, tk, tv, to;
    cudaError_t e;
    if ((e = tchost::make_seq_map(&tq, q, BH, N, DK, C)) != cudaSuccess ||
        (e = tchost::make_seq_map(&tk, k, BH, N, DK, C)) != cudaSuccess ||
        (e = tchost::make_seq_map(&tv, v, BH, N, DK, C)) != cudaSuccess ||
        (e = tchost::make_seq_map(&to, out, BH, N, DK, C)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward: TMA descriptor"};
    int sms = 0;
    if ((e = tchost::sm_count(&sms)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward: device query"};
    const NcPlan pl = plan_noncausal<DK>(sh, seg_chunks, sms);
    if (pl.items > (1LL << 29))
        return {LA_ERR_UNSUPPORTED, cudaSuccess, "la_forward: too many work items"};
    Params p{};
    p.BH = BH;
    p.N = N;
    p.nchunks = pl.nchunks;
    p.nhalf = pl.nhalf;
    p.seg1 = p.grp2 = pl.per;
    p.nseg1 = p.ngrp2 = pl.nseg;
    p.items1 = p.items2 = (int)pl.items;
    p.timeout = 1LL << 32;
    p.phi = sh.phi;
    p.norm = sh.norm;
    // the caller's workspace when given, else a stream-ordered allocation
    void *ws = ws_in;
    if (ws) {
        if (ws_bytes < pl.total)
            return {LA_ERR_INVALID_ARG, cudaSuccess, "la_forward: workspace too small"};
    } else if ((e = tc_workspace_alloc(&ws, pl.total, stream)) != cudaSuccess) {
        return {LA_ERR_NO_MEMORY, e, "la_forward: workspace allocation"};
    }
    char *w8 = static_cast<char *>(ws);
    p.ctrl = reinterpret_cast<int *>(w8);
    p.cnt = reinterpret_cast<int *>(w8 + pl.off_cnt);
    p.part = reinterpret_cast<float *>(w8 + pl.off_part);
    p.status = status;
    e = tc_zero_words(ws, pl.off_part, stream);
    if (e == cudaSuccess) {
        const size_t smem = smem_bytes<DK>();
        auto kern = noncausal_kernel<DK>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e == cudaSuccess) {
            const long long all = 2 * pl.items;
            const int grid = (int)(all < sms ? all : sms);
            e = tchost::launch_dependent(kern, (unsigned)grid, kThreads, smem, stream, tq, tk,
                                         tv, to, p);
            if (e == cudaSuccess) e = cudaGetLastError();
        }
    }
    cudaError_t ef = ws_in ? cudaSuccess : cudaFreeAsync(ws, stream);
    if (e != cudaSuccess) return {LA_ERR_CUDA, e, "la_forward: non-causal kernel launch"};
    if (ef != cudaSuccess) return {LA_ERR_CUDA, ef, "la_forward: workspace free"};
    note_launches(2);  // workspace clear + forward
    return {LA_OK, cudaSuccess, ""};
}

}  // namespace

TcResult launch_noncausal_tc(const void *q, const void *k, const void *v,
                             void *out, const FwdShape &sh, int seg_chunks,
                             int *status, void *ws, size_t ws_bytes,
                             cudaStream_t stream) {
    if (sh.d == 128)
        return launch_noncausal_t<128>(q, k, v, out, sh, seg_chunks, status, ws, ws_bytes, stream);
    return launch_noncausal_t<64>(q, k, v, out, sh, seg_chunks, status, ws, ws_bytes, stream);
}

size_t noncausal_tc_workspace_bytes(const FwdShape &sh, int seg_chunks, int sms) {
    return sh.d == 128 ? plan_noncausal<128>(sh, seg_chunks, sms).total
                       : plan_noncausal<64>(sh, seg_chunks, sms).total;
}

}  // namespace la
