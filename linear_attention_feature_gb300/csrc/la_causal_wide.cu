// Chunkwise causal linear attention for head size d = 128 on tcgen05 tensor
// cores (bf16 in, fp32 accumulate), with optional per-head decay g.  One CTA
// works on all 128 value columns of a (head, segment) item, so every chunk
// is loaded, mapped through phi and multiplied once.
//
// The method ("Linear Attention", chunkwise parallel form; "Story of
// Attention - Part 5", section 6 block formulas, with the normaliser carried
// like the numerator): chunks of C = 128 tokens; for a chunk with local rows
// i, j and S, z the state before it (n = chunk length):
//   P     = phi(Q) phi(K)^T                               (tcgen05 -> TMEM)
//   Pt_ij = P_ij g^(i-j) for j <= i, else 0               (bf16, in TMEM)
//   O     = Pt V + Qhat S,   Qhat_i = g^(i+1) phi(q_i)    (tcgen05)
//   den_i = sum_j Pt_ij + Qhat_i . z                      (CUDA cores)
//   out_i = O_i / den_i
//   S    <- g^n S + Khat^T V,  Khat_t = g^(n-1-t) phi(k_t)  (tcgen05)
//   z    <- g^n z + sum_t Khat_t                          (CUDA cores)
// All four products are single M = 128, N = 128 MMAs per 16-deep K step
// (32 per chunk).  The normaliser is formed on the CUDA cores: the score
// warps sum each row of the bf16-rounded Pt (the exact operand of Pt V),
// and the state warps keep z in fp32 by column sums of Khat and form
// Qhat_i . z.  (A ones column riding along the products would need N = 144
// accumulators and operand blocks that do not fit TMEM and shared memory
// next to two pipeline stages.)
//
// Sequence parallelism: a head's chunks are cut into segments; persistent
// CTAs (one per SM) take (head, segment) items from a ticket counter in
// segment-major order.  A segment with successors first reduces its own
// K and V to its local state (phase A: Khat^T V and sum Khat with weights
// relative to the segment end); its start state is the inclusive prefix
// that its predecessor published, and it publishes its own inclusive prefix
//   incl(s) = g^L incl(s-1) + local(s)
// before running its chunks (phase B).  Every start state is formed by this
// one fixed chain, so results do not depend on timing: repeated calls are
// bit-identical.  The score warps, idle in phase A, fetch the predecessor's
// prefix while phase A runs when it is already published.
//
// Warp roles (576 threads): warp 0 TMA producer (with L2 prefetch two jobs
// ahead), warp 1 MMA issuer and TMEM owner, warps 2-9 feature map (and the
// decay weights), warps 10-13 score epilogue and output epilogue (rows of
// the chunk; outputs stored straight to global memory, 32 bytes per store),
// warps 14-17 state epilogue (bf16 S operand, decay rescale), z, den terms,
// look-back and publication.  Every wait is bounded; a wait that runs out
// sets the device status word to LA_ERR_TIMEOUT and an abort flag, after
// which every wait passes through, so that the kernel finishes (with
// invalid output) instead of hanging.
#include "la_tc.h"
#include "la_tc_host.h"
#include "la_tc_common.cuh"
#include "la_tc_ptx.cuh"

namespace la {
namespace causal_wide {

using namespace la::tc;
using namespace la::tcc;

constexpr int C = 128;  // chunk length (tokens) = MMA M
constexpr int D = 128;  // head size: key features = value columns
constexpr int kWarpT = 2, kNumT = 8, kWarpE1 = 10, kWarpE2 = 14;
constexpr int kThreads = (kWarpE2 + 4) * 32;  // 576
constexpr int kTThreads = kNumT * 32;
constexpr int BAR_T = 1, BAR_E1 = 2, BAR_E2 = 3;
constexpr int STAGES = 2;
constexpr int BLK = C * 128;     // one 64-column SW128 block of a tile (16 KB)
constexpr int TILE = 2 * BLK;    // a [128][128] bf16 tile
constexpr int OFF_Q = 0, OFF_K = TILE, OFF_V = 2 * TILE;
constexpr int STAGE = 3 * TILE;  // 96 KB
// bf16 copy of S (the B operand of Qhat S): MN-major [K = key feature a][N =
// value c], two 64-column blocks of 128 rows
constexpr int OFF_SB = STAGES * STAGE;
constexpr int SB = 2 * BLK;
constexpr int OFF_SMALL = OFF_SB + SB;
constexpr int STATE = D * D + D;  // a published state: S rows (a-major), then z
constexpr int kPrefetch = 3;      // L2 prefetch distance in jobs
// TMEM columns: P in two buffers, O, S
constexpr uint32_t TM_P = 0, TM_O = 256, TM_S = 384, TM_COLS = 512;

struct Params {
    int BH, N, nchunks, seg_chunks, nseg, items;
    float *incl;            // [items][STATE] inclusive prefixes
    int *flags;             // [items]
    float *S_out, *z_out;   // final state [BH][D][D] / [BH][D], or NULL
    int phi, norm;          // elu(x) + 1 on q, k (else identity); divide by den
    int out_v8;             // out is 32-byte aligned (256-bit stores)
    __nv_bfloat16 *out;     // [BH][N][D]
    int *ctrl;              // [0] ticket counter, [1] abort flag
    int *status;            // device status word
    long long timeout;      // clock cycles per bounded wait
};

struct Small {
    float dint[2][C];   // Qhat_i . z per row, by chunk parity (state -> output)
    float z[D];         // running z (state warps)
    float zpark[D];     // z of the predecessor's prefix, fetched early
    float gtab[32];     // g^0 .. g^31 of the current head (score warps)
    // per stage: Q and K (full_qk / empty_qk) and V (full_v / empty_v) are
    // loaded and released separately (Q and K die at Qhat S, V at Pt V)
    uint64_t full_qk[STAGES], empty_qk[STAGES], full_v[STAGES], empty_v[STAGES];
    uint64_t xf[STAGES];
    uint64_t ost_free[2];  // the output epilogue's staging in P buffer b is read
    uint64_t pfull[2], pt_ready[2], pv_done[2];
    uint64_t o_full, o_empty, s_full, sb_ready, lb_done;
    uint64_t khat_ready[2], dint_full[2], dint_empty[2];
    uint64_t item_full[2], item_empty[2];
    uint64_t fin;       // the MMA issuer's last products have completed
    int ring[2];
    int lb_early;       // the predecessor's prefix is parked in TMEM O / zpark
    uint32_t tmem_base;
};

struct Item {
    int bh, seg, c0, c1;
    bool hasA;
};

__device__ __forceinline__ Item decode_item(int t, const Params &p) {
    Item it;
    it.bh = t % p.BH;
    it.seg = t / p.BH;
    it.c0 = it.seg * p.seg_chunks;
    it.c1 = min(it.c0 + p.seg_chunks, p.nchunks);
    it.hasA = it.seg < p.nseg - 1;
    return it;
}

__device__ __forceinline__ int item_index(int bh, int seg, const Params &p) {
    return seg * p.BH + bh;
}

// Pop the next item id from the CTA's item ring (see the producer).
__device__ __forceinline__ int pop_item(Small &sm, int &tl, const Ctx &cx,
                                        int bar_id, int nthreads, bool leader) {
    const int r = tl & 1;
    wait_bar(&sm.item_full[r], (tl >> 1) & 1, cx);
    const int t = ((volatile int *)sm.ring)[r];  // -1 once a wait gave up
    if (bar_id) named_bar_sync(bar_id, nthreads);
    if (leader) mbar_arrive(&sm.item_empty[r]);
    ++tl;
    return t;
}

__device__ __forceinline__ float bf_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf_hi(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// A wait that ignores the abort flag (bounded by the same deadline): used
// at exit, so that no TMA load or MMA is still in flight when the CTA's
// shared memory and TMEM are released.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity, const Ctx &cx) {
    const long long dl = clock64() + cx.timeout;
    while (!mbar_try_wait(bar, parity) && clock64() <= dl) {
    }
}

// ---------------------------------------------------------------- producer

// One job per chunk: phase A jobs load K and V (kept in L2 for phase B),
// phase B jobs load Q, K and V.  Tiles two jobs ahead are prefetched into L2.
__device__ void producer(uint8_t *smem, Small &sm, const Params &p, const Ctx &cx,
                         const CUtensorMap *tq, const CUtensorMap *tk,
                         const CUtensorMap *tv) {
    const uint64_t keep = policy_evict_last(), stream = policy_evict_first(),
                   normal = policy_evict_normal();
    int j = 0, jqk = 0, tl = 0;
    for (;;) {
        int t = atomicAdd(p.ctrl, 1);
        if (t >= p.items || *cx.abort) t = -1;
        const int r = tl & 1;
        wait_bar(&sm.item_empty[r], ((tl >> 1) & 1) ^ 1, cx);
        ((volatile int *)sm.ring)[r] = t;
        mbar_arrive(&sm.item_full[r]);
        ++tl;
        if (t < 0) break;
        const Item it = decode_item(t, p);
        const int nc = it.c1 - it.c0, nA = it.hasA ? nc : 0, nJ = nA + nc;
        if (*cx.abort) continue;  // issue nothing more once a wait gave up
        for (int x = 0; x < nJ + kPrefetch; ++x) {
            if (x < nJ) {  // prefetch of job x, then the load of job x - kPrefetch
                const int pass = x < nA ? 0 : 1;
                const int c = it.c0 + (pass == 0 ? x : x - nA);
                for (int kb = 0; kb < 2; ++kb) {
                    if (pass == 1) tma_prefetch_3d(tq, 64 * kb, c * C, it.bh, normal);
                    tma_prefetch_3d(tk, 64 * kb, c * C, it.bh, pass == 0 ? keep : normal);
                    tma_prefetch_3d(tv, 64 * kb, c * C, it.bh, pass == 0 ? keep : normal);
                }
            }
            const int y = x - kPrefetch;
            if (y < 0) continue;
            const int pass = y < nA ? 0 : 1;
            const int c = it.c0 + (pass == 0 ? y : y - nA);
            const int st = j % STAGES;
            const uint32_t par = ((j / STAGES) & 1) ^ 1;
            uint8_t *base = smem + st * STAGE;
            if (!wait_bar(&sm.empty_qk[st], par, cx)) break;
            mbar_arrive_expect_tx(&sm.full_qk[st], pass == 0 ? TILE : 2 * TILE);
            for (int kb = 0; kb < 2; ++kb) {
                if (pass == 1)
                    tma_load_3d(base + OFF_Q + kb * BLK, tq, &sm.full_qk[st], 64 * kb,
                                c * C, it.bh, stream);
                tma_load_3d(base + OFF_K + kb * BLK, tk, &sm.full_qk[st], 64 * kb, c * C,
                            it.bh, pass == 0 ? keep : stream);
            }
            ++jqk;
            if (!wait_bar(&sm.empty_v[st], par, cx)) break;
            mbar_arrive_expect_tx(&sm.full_v[st], TILE);
            for (int kb = 0; kb < 2; ++kb)
                tma_load_3d(base + OFF_V + kb * BLK, tv, &sm.full_v[st], 64 * kb, c * C,
                            it.bh, pass == 0 ? keep : stream);
            ++j;
        }
    }
    // the last loads of each stage have landed before the CTA may exit
    for (int x = jqk - STAGES; x < jqk; ++x)
        if (x >= 0) drain_wait(&sm.full_qk[x % STAGES], (x / STAGES) & 1, cx);
    for (int x = j - STAGES; x < j; ++x)
        if (x >= 0) drain_wait(&sm.full_v[x % STAGES], (x / STAGES) & 1, cx);
}

// ---------------------------------------------------------------- MMA issuer

// P = phi(Q) phi(K)^T of job `jj` into P buffer nbq & 1, once the chunk is
// transformed and that buffer's previous Pt V has completed.
__device__ __forceinline__ void issue_p(uint8_t *smem, Small &sm, const Ctx &cx,
                                        uint32_t tmem, int jj, int nbq) {
    constexpr uint32_t idP = idesc_bf16(128, 128, 0, 0);
    const int st = jj % STAGES, b = nbq & 1;
    wait_bar(&sm.xf[st], (jj / STAGES) & 1, cx);
    wait_bar(&sm.pv_done[b], ((nbq >> 1) & 1) ^ 1, cx);
    wait_bar(&sm.ost_free[b], ((nbq >> 1) & 1) ^ 1, cx);
    tc_fence_after();
    const uint32_t qb = smem_u32(smem + st * STAGE + OFF_Q);
    const uint32_t kb = smem_u32(smem + st * STAGE + OFF_K);
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
        const uint32_t off = kmajor_off(ks, BLK);
        mma_ss(tmem + TM_P + 128u * b, sdesc_sw128(qb + off, 16, 1024),
               sdesc_sw128(kb + off, 16, 1024), idP, ks > 0 ? 1u : 0u);
    }
    mma_commit(&sm.pfull[b]);
}

// Issues P of B chunk qi+1 now if its feature maps and P buffer are ready.
__device__ __forceinline__ void try_issue_next_p(uint8_t *smem, Small &sm,
                                                 const Ctx &cx, uint32_t tmem,
                                                 int jj, int nbq, int qi, int nB,
                                                 int &p_next) {
    if (p_next != qi + 1 || qi + 1 >= nB) return;
    const int st1 = (jj + 1) % STAGES, b1 = (nbq + 1) & 1;
    if (mbar_try_wait(&sm.xf[st1], ((jj + 1) / STAGES) & 1) &&
        mbar_try_wait(&sm.pv_done[b1], (((nbq + 1) >> 1) & 1) ^ 1) &&
        mbar_try_wait(&sm.ost_free[b1], (((nbq + 1) >> 1) & 1) ^ 1)) {
        issue_p(smem, sm, cx, tmem, jj + 1, nbq + 1);
        ++p_next;
    }
}

template <int kMode>
__device__ void mma_issuer(uint8_t *smem, Small &sm, const Params &p,
                           const Ctx &cx, uint32_t tmem) {
    // Khat^T V: A = Khat^T (MN-major: features contiguous), B = V (MN-major)
    constexpr uint32_t idSU = idesc_bf16(128, 128, 1, 1);
    // Qhat S: A = Qhat (K-major), B = bf16 S (MN-major)
    constexpr uint32_t idQS = idesc_bf16(128, 128, 0, 1);
    // Pt V: A = Pt (TMEM), B = V (MN-major)
    constexpr uint32_t idPV = idesc_bf16(128, 128, 0, 1);
    const uint32_t sb = smem_u32(smem + OFF_SB);
    int j = 0, nb = 0, nsb = 0, no = 0, tl = 0;
    for (;;) {
        const int t = pop_item(sm, tl, cx, 0, 0, true);
        if (t < 0) break;
        const Item it = decode_item(t, p);
        if (it.hasA) {
            // phase A: the segment's local state Khat^T V into S
            for (int c = it.c0; c < it.c1; ++c, ++j) {
                const int st = j % STAGES;
                wait_bar(&sm.xf[st], (j / STAGES) & 1, cx);
                wait_bar(&sm.full_v[st], (j / STAGES) & 1, cx);
                tc_fence_after();
                const uint32_t kb = smem_u32(smem + st * STAGE + OFF_K);
                const uint32_t vb = smem_u32(smem + st * STAGE + OFF_V);
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    mma_ss(tmem + TM_S, sdesc_sw128(kb + ks * 2048, BLK, 1024),
                           sdesc_sw128(vb + ks * 2048, BLK, 1024), idSU,
                           (c > it.c0 || ks > 0) ? 1u : 0u);
                if (c == it.c1 - 1) mma_commit(&sm.s_full);
                mma_commit(&sm.empty_qk[st]);
                mma_commit(&sm.empty_v[st]);
            }
        }
        // phase B.  The state after the item's last chunk is only needed as
        // the sequence's final state; otherwise that chunk has no update.
        const int nB = it.c1 - it.c0;
        const bool final_state = p.S_out && it.seg == p.nseg - 1;
        int p_next = 0;
        for (int qi = 0; qi < nB; ++qi) {
            const int jj = j + qi, nbq = nb + qi;
            const int st = jj % STAGES, b = nbq & 1;
            const bool su = qi + 1 < nB || final_state;
            if (p_next == qi) {
                issue_p(smem, sm, cx, tmem, jj, nbq);
                ++p_next;
            }
            const uint32_t qb = smem_u32(smem + st * STAGE + OFF_Q);
            const uint32_t kb = smem_u32(smem + st * STAGE + OFF_K);
            const uint32_t vb = smem_u32(smem + st * STAGE + OFF_V);
            // the state before this chunk: TMEM S (pre-scaled by g^n) and
            // its bf16 copy; with decay, Qhat and Khat weighted in place
            wait_bar(&sm.sb_ready, nsb & 1, cx);
            ++nsb;
            if (kMode) wait_bar(&sm.khat_ready[nbq & 1], (nbq >> 1) & 1, cx);
            wait_bar(&sm.full_v[st], (jj / STAGES) & 1, cx);
            tc_fence_after();
            if (su) {
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    mma_ss(tmem + TM_S, sdesc_sw128(kb + ks * 2048, BLK, 1024),
                           sdesc_sw128(vb + ks * 2048, BLK, 1024), idSU, 1u);
            }
            try_issue_next_p(smem, sm, cx, tmem, jj, nbq, qi, nB, p_next);
            // O is free once the output epilogue has read the previous chunk's
            wait_bar(&sm.o_empty, (no & 1) ^ 1, cx);
            ++no;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_ss(tmem + TM_O, sdesc_sw128(qb + kmajor_off(ks, BLK), 16, 1024),
                       sdesc_sw128(sb + ks * 2048, BLK, 1024), idQS, ks > 0 ? 1u : 0u);
            // the state warps may now read S and rewrite its bf16 copy; the
            // stage's Q and K are no longer read by the tensor cores
            mma_commit(&sm.s_full);
            mma_commit(&sm.empty_qk[st]);
            // P of the next chunk ahead of Pt V only if Pt is not ready yet
            if (!mbar_try_wait(&sm.pt_ready[b], (nbq >> 1) & 1))
                try_issue_next_p(smem, sm, cx, tmem, jj, nbq, qi, nB, p_next);
            wait_bar(&sm.pt_ready[b], (nbq >> 1) & 1, cx);
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks)
                mma_ts(tmem + TM_O, tmem + TM_P + 128u * b + ks * 8,
                       sdesc_sw128(vb + ks * 2048, BLK, 1024), idPV, 1u);
            mma_commit(&sm.o_full);
            mma_commit(&sm.pv_done[b]);
            mma_commit(&sm.empty_v[st]);
        }
        if (final_state) {
            // S's columns are reused by the next item: wait until the state
            // warps have written the final state out
            wait_bar(&sm.sb_ready, nsb & 1, cx);
            ++nsb;
        }
        j += nB;
        nb += nB;
    }
    // every product has completed before TMEM is released
    mma_commit(&sm.fin);
    drain_wait(&sm.fin, 0, cx);
}

// ---------------------------------------------------------------- transform

template <int kMode>
__device__ void transform(uint8_t *smem, Small &sm, const Params &p,
                          const Ctx &cx, const DecayArgs &dk) {
    const int et = threadIdx.x - kWarpT * 32;  // 0..255
    const int row = et & 127, part = et >> 7;
    int j = 0, nb = 0, tl = 0;
    for (;;) {
        const int t = pop_item(sm, tl, cx, BAR_T, kTThreads, et == 0);
        if (t < 0) break;
        const Item it = decode_item(t, p);
        const float lg = head_log2g(dk, it.bh);
        if (it.hasA) {
            // phase A: Khat_t = g^(L-1-t) phi(k_t), t relative to the segment end
            const int seg_end = min(it.c1 * C, p.N);
            for (int c = it.c0; c < it.c1; ++c, ++j) {
                const int st = j % STAGES;
                wait_bar(&sm.full_qk[st], (j / STAGES) & 1, cx);
                uint8_t *kt = smem + st * STAGE + OFF_K;
                const int tok = c * C + row;
                if (kMode || tok >= p.N) {
                    const float w = tok < p.N ? gpow(lg, seg_end - 1 - tok) : 0.f;
                    transform_row_scaled<D>(kt, row, part, bf2_splat(w), p.phi);
                } else {
                    transform_row<D>(kt, row, part, false, p.phi);
                }
                fence_async_shared();
                named_bar_sync(BAR_T, kTThreads);
                if (et == 0) mbar_arrive(&sm.xf[st]);
            }
        }
        for (int c = it.c0; c < it.c1; ++c, ++j, ++nb) {
            const int st = j % STAGES;
            wait_bar(&sm.full_qk[st], (j / STAGES) & 1, cx);
            uint8_t *qt = smem + st * STAGE + OFF_Q;
            uint8_t *kt = smem + st * STAGE + OFF_K;
            const int n = min(C, p.N - c * C);
            transform_row<D>(qt, row, part, false, p.phi);
            transform_row<D>(kt, row, part, row >= n, p.phi);  // rows past N -> 0
            fence_async_shared();
            named_bar_sync(BAR_T, kTThreads);
            if (et == 0) mbar_arrive(&sm.xf[st]);
            if (kMode) {
                // once P(c) has read the unweighted rows: Khat_t =
                // g^(n-1-t) phi(k_t), Qhat_i = g^(i+1) phi(q_i), in place
                wait_bar(&sm.pfull[nb & 1], (nb >> 1) & 1, cx);
                const float wk = row >= n ? 0.f : gpow(lg, n - 1 - row);
                const float wq = gpow(lg, row + 1);
                scale_row<D>(kt, row, part, bf2_splat(wk));
                scale_row<D>(qt, row, part, bf2_splat(wq));
                fence_async_shared();
                named_bar_sync(BAR_T, kTThreads);
                if (et == 0) mbar_arrive(&sm.khat_ready[nb & 1]);
            }
        }
    }
}

// ---------------------------------------------------------------- score + output

// Causal mask and decay on P (fp32, TMEM), rounded to bf16 in place (the A
// operand of Pt V); returns the row's sum of the rounded values.  One
// thread per row (= TMEM lane).
template <int kMode>
__device__ __forceinline__ float score_chunk(Small &sm, const Ctx &cx, uint32_t lb,
                                             int q, int lane, float lg, int nb,
                                             bool norm) {
    const int b = nb & 1;
    const uint32_t tp = lb + TM_P + 128u * b;
    const int row = q * 32 + lane;
    wait_bar(&sm.pfull[b], (nb >> 1) & 1, cx);
    tc_fence_after();
    float den = 0.f;
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
        uint32_t pk[16];
        if (blk > q) {
#pragma unroll
            for (int e = 0; e < 16; ++e) pk[e] = 0u;
        } else {
            uint32_t v[32];
            tmem_ld32(tp + 32 * blk, v);
            tmem_wait_ld();
            reg_fence(v);
            if (blk < q) {
                if (kMode) {
                    // g^(row - j) = g^(row - 32 blk - 31) g^(31 - e)
                    const float base = gpow(lg, row - 32 * blk - 31);
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        pk[e >> 1] = pack_bf16x2(u2f(v[e]) * (base * sm.gtab[31 - e]),
                                                 u2f(v[e + 1]) * (base * sm.gtab[30 - e]));
                } else {
#pragma unroll
                    for (int e = 0; e < 32; e += 2)
                        pk[e >> 1] = pack_bf16x2(u2f(v[e]), u2f(v[e + 1]));
                }
            } else {
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    // diagonal block: g^(i - j) = g^(lane - e), only where e <= lane
                    float x0 = 0.f, x1 = 0.f;
                    if (e <= lane) x0 = kMode ? u2f(v[e]) * sm.gtab[lane - e] : u2f(v[e]);
                    if (e + 1 <= lane)
                        x1 = kMode ? u2f(v[e + 1]) * sm.gtab[lane - e - 1] : u2f(v[e + 1]);
                    pk[e >> 1] = pack_bf16x2(x0, x1);
                }
            }
            if (norm) {
                float s0 = 0.f, s1 = 0.f;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    s0 += bf_lo(pk[e]);
                    s1 += bf_hi(pk[e]);
                }
                den += s0 + s1;
            }
        }
        tmem_st16(tp + 16 * blk, pk);
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&sm.pt_ready[b]);  // 128 arrivals, one per row
    return den;
}

// One chunk's output: O / den (O alone without the normaliser) in bf16.  O
// is converted into the chunk's P buffer (its Pt is dead once Pt V has
// completed), which frees O for the next chunk's Qhat S at once; the row is
// then read back and stored to global memory (a thread writes its row).
// P of the chunk after next waits for this buffer (ost_free).
__device__ __forceinline__ void output_chunk(Small &sm, const Params &p,
                                             const Ctx &cx, uint32_t lb, int row,
                                             int bh, int c, int nbo, float den_intra,
                                             bool norm) {
    wait_bar(&sm.o_full, nbo & 1, cx);
    tc_fence_after();
    float inv = 1.f;
    if (norm) {
        wait_bar(&sm.dint_full[nbo & 1], (nbo >> 1) & 1, cx);
        inv = 1.f / (den_intra + sm.dint[nbo & 1][row]);
        mbar_arrive(&sm.dint_empty[nbo & 1]);  // 128 arrivals
    }
    const uint32_t tp = lb + TM_P + 128u * (nbo & 1);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint32_t o[32];
        tmem_ld32(lb + TM_O + 32 * g, o);
        tmem_wait_ld();
        reg_fence(o);
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(u2f(o[2 * e]) * inv, u2f(o[2 * e + 1]) * inv);
        tmem_st16(tp + 16 * g, w);
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&sm.o_empty);  // 128 arrivals: O has been read
    const int tok = c * C + row;
    __nv_bfloat16 *dst = p.out + ((size_t)bh * p.N + tok) * D;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t w[32];
        tmem_ld32(tp + 32 * h, w);
        tmem_wait_ld();
        reg_fence(w);
        if (tok < p.N) {
            if (p.out_v8) {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    st_v8(dst + 64 * h + 16 * u, *reinterpret_cast<const uint32_t(*)[8]>(w + 8 * u));
            } else {
                uint4 *d4 = reinterpret_cast<uint4 *>(dst + 64 * h);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    d4[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
            }
        }
    }
    tc_fence_before();
    mbar_arrive(&sm.ost_free[nbo & 1]);  // 128 arrivals
}

template <int kMode>
__device__ void score_output(Small &sm, const Params &p, const Ctx &cx,
                             const DecayArgs &dk, uint32_t tmem) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3, row = q * 32 + lane;
    const int et = threadIdx.x - kWarpE1 * 32;
    const uint32_t lb = tmem + ((uint32_t)(q * 32) << 16);
    const bool norm = p.norm != 0;
    int nb = 0, tl = 0;
    for (;;) {
        const int t = pop_item(sm, tl, cx, BAR_E1, 128, et == 0);
        if (t < 0) break;
        const Item it = decode_item(t, p);
        const float lg = head_log2g(dk, it.bh);
        if (kMode && et < 32) sm.gtab[et] = gpow(lg, et);
        // The predecessor's inclusive prefix, if it is already published,
        // fetched now (phase A runs meanwhile) into TMEM O (row `row` of S)
        // and zpark; the state warps take it from there.
        if (et == 0)
            sm.lb_early = (it.hasA && it.seg > 0 &&
                           load_flag(p.flags + item_index(it.bh, it.seg - 1, p)) >= FLAG_INCL)
                              ? 1 : 0;
        named_bar_sync(BAR_E1, 128);
        if (sm.lb_early) {
            const float *src = p.incl + (size_t)item_index(it.bh, it.seg - 1, p) * STATE;
#pragma unroll 1
            for (int g = 0; g < 4; ++g) {
                float x[32];
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    ld_cg_v8(src + row * D + 32 * g + 8 * u,
                             *reinterpret_cast<float(*)[8]>(x + 8 * u));
                uint32_t w[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(x[e]);
                tmem_st32(lb + TM_O + 32 * g, w);
            }
            sm.zpark[row] = __ldcg(src + D * D + row);
            tmem_wait_st();
        }
        tc_fence_before();
        named_bar_sync(BAR_E1, 128);
        if (et == 0) mbar_arrive(&sm.lb_done);
        // phase B: the output of chunk c - 1 (its O completes before P of
        // chunk c, issued after it), then the scores of chunk c
        int pend = -1, pend_c = 0;
        float pend_den = 0.f;
        for (int c = it.c0; c < it.c1; ++c, ++nb) {
            if (pend >= 0)
                output_chunk(sm, p, cx, lb, row, it.bh, pend_c, pend, pend_den, norm);
            pend_den = score_chunk<kMode>(sm, cx, lb, q, lane, lg, nb, norm);
            pend = nb;
            pend_c = c;
        }
        if (pend >= 0) output_chunk(sm, p, cx, lb, row, it.bh, pend_c, pend, pend_den, norm);
    }
}

// ---------------------------------------------------------------- state

// Column sums of two adjacent key features (2 pr, 2 pr + 1) of a [128][128]
// bf16 SW128 tile: this thread sums the 64 rows of half `hf` (in an order
// that keeps the two halves of a warp on different banks), then adds its
// partner lane's half.
__device__ __forceinline__ void colsum(const uint8_t *tile, int pr, int hf,
                                       float &s0, float &s1) {
    const int f = 2 * pr;
    const uint8_t *blk = tile + (f >> 6) * BLK;
    const int col = f & 63, ch = col >> 3, cb = (col & 7) * 2;
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll 8
    for (int s = 0; s < 64; s += 2) {
        const int t0 = hf * 64 + ((s + 4 * hf) & 63);
        const int t1 = hf * 64 + ((s + 1 + 4 * hf) & 63);
        const uint32_t x0 = *reinterpret_cast<const uint32_t *>(
            blk + t0 * 128 + ((ch ^ (t0 & 7)) << 4) + cb);
        const uint32_t x1 = *reinterpret_cast<const uint32_t *>(
            blk + t1 * 128 + ((ch ^ (t1 & 7)) << 4) + cb);
        a0 += bf_lo(x0);
        a1 += bf_hi(x0);
        b0 += bf_lo(x1);
        b1 += bf_hi(x1);
    }
    a0 += b0;
    a1 += b1;
    s0 = a0 + __shfl_xor_sync(~0u, a0, 1);
    s1 = a1 + __shfl_xor_sync(~0u, a1, 1);
}

// Row a of a [128][128] bf16 SW128 tile dotted with z (fp32, shared memory).
__device__ __forceinline__ float dot_row(const uint8_t *tile, int a, const float *z) {
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int cc = 0; cc < 16; ++cc) {
        const uint4 x = *reinterpret_cast<const uint4 *>(
            tile + (cc >> 3) * BLK + sw128_offset(a, (cc & 7) * 8));
        const float4 z0 = *reinterpret_cast<const float4 *>(z + cc * 8);
        const float4 z1 = *reinterpret_cast<const float4 *>(z + cc * 8 + 4);
        acc0 = fmaf(bf_lo(x.x), z0.x, acc0);
        acc1 = fmaf(bf_hi(x.x), z0.y, acc1);
        acc0 = fmaf(bf_lo(x.y), z0.z, acc0);
        acc1 = fmaf(bf_hi(x.y), z0.w, acc1);
        acc0 = fmaf(bf_lo(x.z), z1.x, acc0);
        acc1 = fmaf(bf_hi(x.z), z1.y, acc1);
        acc0 = fmaf(bf_lo(x.w), z1.z, acc0);
        acc1 = fmaf(bf_hi(x.w), z1.w, acc1);
    }
    return acc0 + acc1;
}

// 32 values of row a, columns [32 g, 32 g + 32), into the bf16 S operand.
__device__ __forceinline__ void store_sb32(uint8_t *sb, int a, int g, const float (&x)[32]) {
    uint8_t *blk = sb + (g >> 1) * BLK;
    const int c0 = 32 * (g & 1);
#pragma unroll
    for (int ch = 0; ch < 4; ++ch)
        *reinterpret_cast<uint4 *>(blk + sw128_offset(a, c0 + ch * 8)) =
            make_uint4(pack_bf16x2(x[8 * ch], x[8 * ch + 1]),
                       pack_bf16x2(x[8 * ch + 2], x[8 * ch + 3]),
                       pack_bf16x2(x[8 * ch + 4], x[8 * ch + 5]),
                       pack_bf16x2(x[8 * ch + 6], x[8 * ch + 7]));
}

template <int kMode>
__device__ void state_role(uint8_t *smem, Small &sm, const Params &p, const Ctx &cx,
                           const DecayArgs &dk, uint32_t tmem) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;
    const int et = threadIdx.x - kWarpE2 * 32;
    const int a = q * 32 + lane;          // TMEM lane: state row, and output row
    const int pr = et >> 1, hf = et & 1;  // column sums: feature pair, token half
    const int fz = 2 * pr + hf;           // the z entry this thread updates
    const uint32_t lb = tmem + ((uint32_t)(q * 32) << 16);
    uint8_t *sb = smem + OFF_SB;
    const bool norm = p.norm != 0;
    const bool track_z = norm || p.S_out;
    int j = 0, nb = 0, ns = 0, nl = 0, tl = 0;
    for (;;) {
        const int t = pop_item(sm, tl, cx, BAR_E2, 128, et == 0);
        if (t < 0) break;
        const Item it = decode_item(t, p);
        const float lg = head_log2g(dk, it.bh);
        const float gL = gpow(lg, p.seg_chunks * C);
        const float f0 = gpow(lg, min(C, p.N - it.c0 * C));
        float zA = 0.f;  // phase A: entry fz of the segment's local z
        if (it.hasA) {
            for (int c = it.c0; c < it.c1; ++c, ++j) {
                const int st = j % STAGES;
                wait_bar(&sm.xf[st], (j / STAGES) & 1, cx);
                float s0, s1;
                colsum(smem + st * STAGE + OFF_K, pr, hf, s0, s1);
                zA += hf ? s1 : s0;
                named_bar_sync(BAR_E2, 128);
                if (et == 0) mbar_arrive(&sm.empty_qk[st]);
            }
            wait_bar(&sm.s_full, ns & 1, cx);
            ++ns;
            tc_fence_after();
        }
        // The start state is the predecessor's inclusive prefix: parked by
        // the score warps, or read here once published.
        wait_bar(&sm.lb_done, nl & 1, cx);
        ++nl;
        tc_fence_after();
        const bool pred = it.seg > 0;
        const bool early = sm.lb_early != 0;
        const float *src =
            pred ? p.incl + (size_t)item_index(it.bh, it.seg - 1, p) * STATE : nullptr;
        if (pred && !early) {
            if (warp == kWarpE2 && lane == 0)
                poll_flag_at_least(p.flags + item_index(it.bh, it.seg - 1, p), FLAG_INCL,
                                   FLAG_INCL, cx);
            named_bar_sync(BAR_E2, 128);
        }
        float *dst = it.hasA ? p.incl + (size_t)t * STATE : nullptr;
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {
            float pv[32];
            if (!pred) {
#pragma unroll
                for (int e = 0; e < 32; ++e) pv[e] = 0.f;
            } else if (early) {
                uint32_t v[32];
                tmem_ld32(lb + TM_O + 32 * g, v);
                tmem_wait_ld();
                reg_fence(v);
#pragma unroll
                for (int e = 0; e < 32; ++e) pv[e] = u2f(v[e]);
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    ld_cg_v8(src + a * D + 32 * g + 8 * u,
                             *reinterpret_cast<float(*)[8]>(pv + 8 * u));
            }
            if (it.hasA) {
                // incl(s) = g^L incl(s-1) + local(s)
                uint32_t v[32];
                tmem_ld32(lb + TM_S + 32 * g, v);
                tmem_wait_ld();
                reg_fence(v);
                float4 *d4 = reinterpret_cast<float4 *>(dst + a * D + 32 * g);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    d4[u] = make_float4(fmaf(gL, pv[4 * u], u2f(v[4 * u])),
                                        fmaf(gL, pv[4 * u + 1], u2f(v[4 * u + 1])),
                                        fmaf(gL, pv[4 * u + 2], u2f(v[4 * u + 2])),
                                        fmaf(gL, pv[4 * u + 3], u2f(v[4 * u + 3])));
            }
            store_sb32(sb, a, g, pv);
            // phase-B start: TMEM S = g^n0 S_start
            uint32_t w[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(f0 * pv[e]);
            tmem_st32(lb + TM_S + 32 * g, w);
        }
        sm.z[a] = pred ? (early ? sm.zpark[a] : __ldcg(src + D * D + a)) : 0.f;
        tmem_wait_st();
        named_bar_sync(BAR_E2, 128);
        if (it.hasA) {
            dst[D * D + fz] = fmaf(gL, sm.z[fz], zA);
            __threadfence();
        }
        fence_async_shared();
        tc_fence_before();
        named_bar_sync(BAR_E2, 128);
        if (et == 0) {
            if (it.hasA) publish_flag(p.flags + t, FLAG_INCL);
            mbar_arrive(&sm.sb_ready);
        }
        // phase B
        for (int c = it.c0; c < it.c1; ++c, ++j, ++nb) {
            const int st = j % STAGES;
            const int n = min(C, p.N - c * C);
            uint8_t *stage = smem + st * STAGE;
            wait_bar(&sm.xf[st], (j / STAGES) & 1, cx);
            if (kMode) wait_bar(&sm.khat_ready[nb & 1], (nb >> 1) & 1, cx);
            if (track_z) {
                // den term of this chunk from z before it, then z after it
                if (norm) {
                    const float di = dot_row(stage + OFF_Q, a, sm.z);
                    wait_bar(&sm.dint_empty[nb & 1], ((nb >> 1) & 1) ^ 1, cx);
                    sm.dint[nb & 1][a] = di;
                }
                float s0, s1;
                colsum(stage + OFF_K, pr, hf, s0, s1);
                named_bar_sync(BAR_E2, 128);  // z read, den terms written
                if (et == 0) {
                    if (norm) mbar_arrive(&sm.dint_full[nb & 1]);
                    mbar_arrive(&sm.empty_qk[st]);
                }
                sm.z[fz] = fmaf(kMode ? gpow(lg, n) : 1.f, sm.z[fz], hf ? s1 : s0);
                named_bar_sync(BAR_E2, 128);
            } else {
                named_bar_sync(BAR_E2, 128);
                if (et == 0) mbar_arrive(&sm.empty_qk[st]);
            }
            wait_bar(&sm.s_full, ns & 1, cx);
            ++ns;
            tc_fence_after();
            if (c + 1 < it.c1) {
                // the bf16 copy of S for chunk c+1, and with decay the
                // rescale g^n of the accumulator
                const float f = gpow(lg, min(C, p.N - (c + 1) * C));
#pragma unroll 1
                for (int g = 0; g < 4; ++g) {
                    uint32_t v[32];
                    tmem_ld32(lb + TM_S + 32 * g, v);
                    tmem_wait_ld();
                    reg_fence(v);
                    float x[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[e] = u2f(v[e]);
                    store_sb32(sb, a, g, x);
                    if (kMode) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(f * x[e]);
                        tmem_st32(lb + TM_S + 32 * g, v);
                    }
                }
                if (kMode) tmem_wait_st();
                fence_async_shared();
                tc_fence_before();
                named_bar_sync(BAR_E2, 128);
                if (et == 0) mbar_arrive(&sm.sb_ready);
            }
        }
        if (p.S_out && it.seg == p.nseg - 1) {
            // the state after the sequence's last token (a decode continues
            // from it); the last chunk's update ran
#pragma unroll 1
            for (int g = 0; g < 4; ++g) {
                uint32_t v[32];
                tmem_ld32(lb + TM_S + 32 * g, v);
                tmem_wait_ld();
                reg_fence(v);
                float4 *d4 = reinterpret_cast<float4 *>(p.S_out + ((size_t)it.bh * D + a) * D + 32 * g);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    d4[u] = make_float4(u2f(v[4 * u]), u2f(v[4 * u + 1]), u2f(v[4 * u + 2]),
                                        u2f(v[4 * u + 3]));
            }
            p.z_out[(size_t)it.bh * D + a] = sm.z[a];
            tc_fence_before();
            named_bar_sync(BAR_E2, 128);
            if (et == 0) mbar_arrive(&sm.sb_ready);
        }
    }
}

// ---------------------------------------------------------------- kernel

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
causal_wide_kernel(const __grid_constant__ CUtensorMap tq,
                   const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const Params p,
                   const DecayArgs dk) {
    extern __shared__ __align__(1024) uint8_t smem[];
    // The 128-byte swizzle needs 1024-byte aligned tiles, and the layout
    // fills the shared memory a CTA may have, with no room for padding.
    if (smem_u32(smem) & 1023u) {
        if (threadIdx.x == 0 && atomicCAS(p.status, 0, (int)LA_ERR_UNSUPPORTED) == 0)
            atomicExch(p.status + 1, (int)((blockIdx.x << 20) | 0xA1160u));
        return;
    }
    Small &sm = *reinterpret_cast<Small *>(smem + OFF_SMALL);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Ctx cx{reinterpret_cast<volatile int *>(p.ctrl + 1), p.status, p.timeout};
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sm.full_qk[s], 1);
            mbar_init(&sm.full_v[s], 1);
            mbar_init(&sm.empty_qk[s], 2);  // MMA commit + state warps
            mbar_init(&sm.empty_v[s], 1);
            mbar_init(&sm.xf[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.pfull[b], 1);
            mbar_init(&sm.pt_ready[b], 128);
            mbar_init(&sm.pv_done[b], 1);
            mbar_init(&sm.khat_ready[b], 1);
            mbar_init(&sm.dint_full[b], 1);
            mbar_init(&sm.dint_empty[b], 128);
            mbar_init(&sm.ost_free[b], 128);
            mbar_init(&sm.item_full[b], 1);
            mbar_init(&sm.item_empty[b], 4);
        }
        mbar_init(&sm.o_full, 1);
        mbar_init(&sm.o_empty, 128);
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.sb_ready, 1);
        mbar_init(&sm.lb_done, 1);
        mbar_init(&sm.fin, 1);
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(&sm.tmem_base, TM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tq);
        tma_prefetch_desc(&tk);
        tma_prefetch_desc(&tv);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        if (lane == 0) producer(smem, sm, p, cx, &tq, &tk, &tv);
    } else if (warp == 1) {
        if (lane == 0) mma_issuer<kMode>(smem, sm, p, cx, tmem);
    } else if (warp < kWarpE1) {
        transform<kMode>(smem, sm, p, cx, dk);
    } else if (warp < kWarpE2) {
        score_output<kMode>(sm, p, cx, dk, tmem);
    } else {
        state_role<kMode>(smem, sm, p, cx, dk, tmem);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TM_COLS);
}

constexpr size_t kSmemBytes = (size_t)OFF_SMALL + sizeof(Small);
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(OFF_SB % 1024 == 0 && STAGE % 1024 == 0, "SW128 tiles need 1024-byte alignment");

}  // namespace causal_wide

namespace {

inline size_t align_up_w(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Work decomposition and workspace layout of one launch.
struct WidePlan {
    int seg_chunks, nseg, nchunks;
    long long items;
    size_t off_flags, off_incl, total;
};

WidePlan plan_wide(const FwdShape &sh, int seg_chunks, int sms) {
    using namespace causal_wide;
    WidePlan pl{};
    pl.nchunks = (sh.N + C - 1) / C;
    if (seg_chunks <= 0) seg_chunks = wide_segment_chunks(sh.BH(), pl.nchunks, sms);
    if (seg_chunks > pl.nchunks) seg_chunks = pl.nchunks;
    pl.seg_chunks = seg_chunks;
    pl.nseg = (pl.nchunks + seg_chunks - 1) / seg_chunks;
    pl.items = sh.BH() * pl.nseg;
    pl.off_flags = 256;
    pl.off_incl = align_up_w(pl.off_flags + sizeof(int) * (size_t)pl.items, 256);
    pl.total = pl.off_incl +
               (pl.nseg > 1 ? sizeof(float) * (size_t)STATE * (size_t)pl.items : 0);
    return pl;
}

TcResult launch_wide_with(const void *q, const void *k, const void *v, void *out,
                          const FwdShape &sh, const DecayArgs &dk, const WidePlan &pl,
                          int *status, char *ws, float *S_out, float *z_out,
                          cudaStream_t stream, int sms) {
    using namespace causal_wide;
    const int BH = (int)sh.BH(), N = sh.N;
    CUtensorMap tq, tk, tv;
    cudaError_t e;
    if ((e = tchost::make_seq_map(&tq, q, BH, N, D, C)) != cudaSuccess ||
        (e = tchost::make_seq_map(&tk, k, BH, N, D, C)) != cudaSuccess ||
        (e = tchost::make_seq_map(&tv, v, BH, N, D, C)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward: TMA descriptor"};
    Params p{};
    p.BH = BH;
    p.N = N;
    p.nchunks = pl.nchunks;
    p.seg_chunks = pl.seg_chunks;
    p.nseg = pl.nseg;
    p.items = (int)pl.items;
    p.timeout = 1LL << 32;
    p.S_out = S_out;
    p.z_out = z_out;
    p.phi = sh.phi;
    p.norm = sh.norm;
    p.out = static_cast<__nv_bfloat16 *>(out);
    p.out_v8 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
    p.ctrl = reinterpret_cast<int *>(ws);
    p.flags = reinterpret_cast<int *>(ws + pl.off_flags);
    p.incl = reinterpret_cast<float *>(ws + pl.off_incl);
    p.status = status;
    // the ticket counter, abort flag and segment flags start at zero; the
    // published states need no clearing
    if ((e = tc_zero_words(ws, pl.off_incl, stream)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward: workspace clear"};
    auto kern = dk.has ? causal_wide_kernel<1> : causal_wide_kernel<0>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kSmemBytes)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward: kernel attribute"};
    const int grid = (int)(pl.items < sms ? pl.items : sms);
    kern<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p, dk);
    if ((e = cudaGetLastError()) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward: causal kernel launch"};
    note_launches(2);  // workspace clear + forward
    return {LA_OK, cudaSuccess, ""};
}

}  // namespace

// Segment length for the d = 128 kernel: the wave rule (per-item overhead
// of about three chunk times), with segments capped so that the K and V a
// wave reads in phase A (SMs x length x 64 KB) stay in L2 until phase B
// reads them again.
int wide_segment_chunks(long long heads, int nchunks, int sms) {
    constexpr int kCap = 8;
    int best = nchunks < kCap ? nchunks : kCap;
    long long best_cost = -1;
    if (sms < 1) sms = 1;
    for (int len = best; len >= 1; --len) {
        const long long nseg = (nchunks + len - 1) / len;
        const long long waves = (heads * nseg + sms - 1) / sms;
        const long long cost = waves * (2 * len + (nseg > 1 ? 3 : 0));
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = len;
        }
    }
    return best;
}

TcResult launch_causal_wide(const void *q, const void *k, const void *v, void *out,
                            const FwdShape &sh, const DecayArgs &dk, int seg_chunks,
                            int *status, void *ws_in, size_t ws_bytes, float *S_out,
                            float *z_out, cudaStream_t stream) {
    int sms = 0;
    cudaError_t e;
    if ((e = tchost::sm_count(&sms)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward: device query"};
    const WidePlan pl = plan_wide(sh, seg_chunks, sms);
    if (pl.items > (1LL << 30))
        return {LA_ERR_UNSUPPORTED, cudaSuccess, "la_forward: too many work items"};
    void *ws = ws_in;
    if (ws) {
        if (ws_bytes < pl.total)
            return {LA_ERR_INVALID_ARG, cudaSuccess, "la_forward: workspace too small"};
    } else if ((e = cudaMallocAsync(&ws, pl.total, stream)) != cudaSuccess) {
        return {LA_ERR_NO_MEMORY, e, "la_forward: workspace allocation"};
    }
    TcResult r = launch_wide_with(q, k, v, out, sh, dk, pl, status, static_cast<char *>(ws),
                                  S_out, z_out, stream, sms);
    if (!ws_in) {
        cudaError_t ef = cudaFreeAsync(ws, stream);
        if (r.status == LA_OK && ef != cudaSuccess)
            return {LA_ERR_CUDA, ef, "la_forward: workspace free"};
    }
    return r;
}

size_t causal_wide_workspace_bytes(const FwdShape &sh, int seg_chunks, int sms) {
    return plan_wide(sh, seg_chunks, sms).total;
}

TcResult launch_causal_wide_fixed(const void *q, const void *k, const void *v,
                                  void *out, const FwdShape &sh, const DecayArgs &dk,
                                  int *status, char *scratch, size_t cap,
                                  cudaStream_t stream) {
    int sms = 0;
    cudaError_t e;
    if ((e = tchost::sm_count(&sms)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward_causal_noalloc: device query"};
    // lengthen segments until the workspace fits the fixed scratch
    WidePlan pl = plan_wide(sh, 0, sms);
    while (pl.total > cap && pl.seg_chunks < pl.nchunks)
        pl = plan_wide(sh, pl.seg_chunks * 2 < pl.nchunks ? pl.seg_chunks * 2 : pl.nchunks, sms);
    if (pl.total > cap || pl.items > (1LL << 30))
        return {LA_ERR_UNSUPPORTED, cudaSuccess,
                "la_forward_causal_noalloc: the problem needs more workspace "
                "than the 16 MiB static scratch holds (too many heads)"};
    return launch_wide_with(q, k, v, out, sh, dk, pl, status, scratch, nullptr, nullptr,
                            stream, sms);
}

}  // namespace la
