// Chunkwise causal linear attention for head size d = 128 on tcgen05 tensor
// cores (bf16 in, fp32 accumulate), with optional per-head decay g.  One CTA
// works on all 128 value columns of a (head, segment) item, so every chunk
// is loaded, mapped through phi and multiplied once.
//
// The method ("Linear Attention", chunkwise parallel form; "Story of
// Attention - Part 5", section 6 block formulas, with the normaliser carried
// like the numerator): chunks of C = 128 tokens; for a chunk with local rows
// i, j and S, z the state before it (n = chunk length):
//   P        = phi(Q) phi(K)^T                            (tcgen05 -> TMEM)
//   Pt_ij    = P_ij g^(i-j) for j <= i, else 0            (bf16, in TMEM)
//   O | den  = Pt [V | 1] + Qhat [S | z],  Qhat_i = g^(i+1) phi(q_i)
//   out_i    = O_i / den_i
//   S | z   <- g^n [S | z] + Khat^T [V | 1],  Khat_t = g^(n-1-t) phi(k_t)
// The normaliser rides along as a 129th column of the products (N = 144):
// [V | 1] ends in a block whose column 0 is one, [S | z] in a block holding
// z, so numerator and denominator come from the same bf16 operands.
//
// Decay modes.  Mode 1 computes P from the unweighted phi(Q), phi(K) and
// weights the rows in place once P has read them (K rows in shared memory,
// Q rows in TMEM).  Mode 2, used with the elu + 1 map (positive features)
// when every decay is at least 0.77, weights both operands as soon as they
// are mapped: Khat_j = g^(n-1-j) phi(k_j) and Q'_i = g^(i+1-n) phi(q_i), so
// that P = Q' Khat^T is already g^(i-j) phi(q_i) . phi(k_j) (only the mask
// remains), while the bf16 state operand carries g^n: Q' (g^n [S | z]) =
// Qhat [S | z].  No product waits for a weighting pass, and the powers stay
// in range for such decays (g^-(C-1) <= 2^48 in Q', P's masked entries up
// to g^-(C-1) times a score).
//
// Memory plan.  TMEM (480 of 512 columns): P (single buffer, Pt written
// back in place), O | den (144), S | z (144) and phi(Q) (64 columns of bf16
// pairs: the A operand of P and of Qhat [S | z], so Q needs no shared-memory
// stage, only a landing slot that the feature map empties into TMEM).
// Shared memory (224 KB): the bf16 [S | z] operand (48 KB), the Q landing
// slot, two K stages, two V stages and one ones block shared by both V
// stages -- each V stage's two 64-column blocks sit at a distance (the
// descriptor's leading byte offset) that puts its third block on the ones.
//
// Sequence parallelism: a head's chunks are cut into segments; persistent
// CTAs (one per SM) take (head, segment) items from a ticket counter in
// segment-major order.  Segment 0 starts from the zero state and runs the
// chunk loop (phase B) at once.  A later segment s first reduces its
// predecessor's K and V to that segment's local state (phase A:
// Khat^T [V | 1] with weights relative to the end of that range, its own
// start), keeps it in TMEM as the first term of its start state, and
// publishes it when a later segment needs it.  The other terms are the
// states published by segments 1 .. s-1 (the local states of segments
// s-2 .. 0):
//   start(s) = local(s-1) + sum_{m = 2..s} g^(L (m - 1)) local(s - m),
// added in this fixed order, so results do not depend on timing (repeated
// calls are bit-identical) and no segment waits on another's look-back.
// The score warps, idle in phase A, form the published part while phase A
// runs when its segments have already published.
//
// Warp roles (576 threads): warp 0 TMA producer (with L2 prefetch ahead),
// warp 1 MMA issuer and TMEM owner, warps 2-9 feature map (phi(K) in place,
// phi(Q) into TMEM; the decay weights), warps 10-13 score and output
// epilogues, warps 14-17 state epilogue (bf16 [S | z] operand, decay
// rescale), look-back and publication.  Per chunk the tensor pipe runs
// P, Khat^T [V | 1], Qhat [S | z], Pt [V | 1].  Every wait is bounded; a wait
// that runs out sets the device status word to LA_ERR_TIMEOUT and an abort
// flag, after which every wait passes through, so that the kernel finishes
// (with invalid output) instead of hanging.
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
constexpr int NX = D + 16;  // N of the products that carry the normaliser
constexpr int kWarpT = 2, kNumT = 8, kWarpE1 = 10, kWarpE2 = 14;
constexpr int kThreads = (kWarpE2 + 4) * 32;  // 576
constexpr int kTThreads = kNumT * 32;
constexpr int BAR_T = 1, BAR_E1 = 2, BAR_E2 = 3;
constexpr int STAGES = 2;
constexpr int BLK = C * 128;   // one 64-column SW128 block of 128 rows (16 KB)
constexpr int TILE = 2 * BLK;  // a [128][128] bf16 tile
// shared memory (byte offsets)
constexpr int OFF_SB = 0;                  // [S | z]: S block 0, S block 1, z block
constexpr int OFF_Q = 3 * BLK;             // Q landing slot
constexpr int OFF_K0 = OFF_Q + TILE;       // K, stage 0
constexpr int OFF_V1 = OFF_K0 + TILE;      // V stage 1, block 0
constexpr int OFF_K1 = OFF_V1 + BLK;       // K, stage 1
constexpr int OFF_V0 = OFF_K1 + TILE + BLK;  // V stage 0, blocks 0 and 1
constexpr int OFF_ONES = OFF_V0 + TILE;    // [V | 1]'s ones block (column 0 = 1)
constexpr int LBO_V0 = BLK, LBO_V1 = 3 * BLK;
static_assert(OFF_V1 + LBO_V1 == OFF_K1 + TILE, "V stage 1 block 1 placement");
static_assert(OFF_V0 + 2 * LBO_V0 == OFF_ONES && OFF_V1 + 2 * LBO_V1 == OFF_ONES,
              "both V stages must reach the ones block through their LBO");
constexpr int OFF_SMALL = OFF_ONES + BLK;  // 224 KB
// A published state: S, then z.  S is stored so that the 32 lanes of a warp
// (32 consecutive rows a) move 512 contiguous bytes per access: float4
// number u of the 32-column group g of row a sits at float4 index
// (8 g + u) * 128 + a.
constexpr int STATE = D * D + D;
constexpr int kPrefetch = 1;      // phase-A L2 prefetch distance in jobs
constexpr float kFoldMin = 0.77f;  // smallest decay for the folded-weights mode
// TMEM columns
constexpr uint32_t TM_P = 0, TM_O = 128, TM_S = 272, TM_Q = 416, TM_COLS = 512;

__host__ __device__ constexpr int k_off(int st) { return st ? OFF_K1 : OFF_K0; }
__host__ __device__ constexpr int v_off(int st) { return st ? OFF_V1 : OFF_V0; }
__host__ __device__ constexpr int v_lbo(int st) { return st ? LBO_V1 : LBO_V0; }

struct Params {
    int BH, N, nchunks, seg_chunks, nseg, items;
    int seg0;               // chunks of segment 0 (later segments: seg_chunks)
    float *agg;             // [items][STATE] each segment's local state
    int *flags;             // [items]
    float *S_out, *z_out;   // final state [BH][D][D] / [BH][D], or NULL
    int phi, norm;          // elu(x) + 1 on q, k (else identity); divide by den
    int *ctrl;              // [0] ticket counter, [1] abort flag
    int *status;            // device status word
    long long timeout;      // clock cycles per bounded wait
    int hold_seg;           // test hook: this segment never publishes (-1: none)
};

struct Small {
    float gtab[32];  // g^0 .. g^31 of the current head (score warps)
    uint64_t q_full, q_empty;                       // Q landing slot
    uint64_t k_full[STAGES], k_empty[STAGES], v_full[STAGES], v_empty[STAGES];
    uint64_t xfk[STAGES];  // phi(K) (or Khat) ready in the stage
    uint64_t xfq;          // phi(Q) written to TMEM
    uint64_t q_free;       // phi(Q)'s TMEM columns read by the chunk's last product
    uint64_t khat_ready;   // with decay: Khat and Qhat weighted in place
    uint64_t pfull, pt_ready, pv_done;
    uint64_t o_full, o_empty, s_full, sb_ready, lb_done;
    uint64_t item_full[2], item_empty[2];
    uint64_t fin;
    int ring[2];
    int lb_early;  // the start state is parked in TMEM O (S, and z in column D)
    uint32_t tmem_base;
};

// A work item: segment `seg` of head `bh`, chunks [c0, c1) (segment 0
// spans seg0 chunks, later ones seg_chunks).  Phase A of segment s >= 1
// reduces its predecessor's chunks [a0, a1 = c0) to that segment's local
// state, weighted relative to c0: the first term of its own start state,
// kept in TMEM, published (pub) when a later segment needs it too.
// Segment 0 starts from zero and runs phase B at once.
struct Item {
    int bh, seg, c0, c1, a0, a1;
    bool hasA, pub;
};

__device__ __forceinline__ Item decode_item(int t, const Params &p) {
    Item it;
    it.bh = t % p.BH;
    it.seg = t / p.BH;
    it.c0 = it.seg == 0 ? 0 : p.seg0 + (it.seg - 1) * p.seg_chunks;
    it.c1 = min(it.seg == 0 ? p.seg0 : it.c0 + p.seg_chunks, p.nchunks);
    it.a0 = it.seg <= 1 ? 0 : p.seg0 + (it.seg - 2) * p.seg_chunks;
    it.a1 = it.c0;
    it.hasA = it.seg > 0;
    it.pub = it.seg > 0 && it.seg < p.nseg - 1;
    return it;
}

__device__ __forceinline__ int item_index(int bh, int seg, const Params &p) {
    return seg * p.BH + bh;
}

// Pop the next item id from the CTA's item ring (see the producer).
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

// ---------------------------------------------------------------- look-back

// True once segments 1 .. seg-1 of head bh (which hold the local states of
// segments 0 .. seg-2) have all published (one warp; 32 flags per look).
// Without `wait` it looks once.
__device__ __forceinline__ bool preds_published(const Params &p, const Ctx &cx, int bh,
                                                int seg, int lane, bool wait) {
    long long dl = 0;
    for (int base = 1; base < seg; base += 32) {
        const int s = base + lane;
        const int fi = item_index(bh, s < seg ? s : 1, p);
        const bool ok = LA_DCHECK(p.status, fi >= 0 && fi < p.items);
        const int *fp = p.flags + (ok ? fi : 0);
        for (;;) {
            const int f = s < seg && ok ? load_flag(fp) : FLAG_AGG;
            if (__all_sync(~0u, f >= FLAG_AGG)) break;
            if (!wait) return false;
            if (__any_sync(~0u, *cx.abort != 0)) return false;
            const long long now = __shfl_sync(~0u, clock64(), 0);
            if (dl == 0) {
                dl = now + cx.timeout;
            } else if (now > dl) {
                if (lane == 0)
                    raise_timeout(cx, 0x80000u | ((uint32_t)(reinterpret_cast<uintptr_t>(fp) >> 2) & 0x7FFFFu));
                return false;
            }
            __nanosleep(64);
        }
    }
    return true;
}

// Row r of the published part of the start state, columns [32 g, 32 g + 32)
// (g < 4) or z[r] in acc[0] (g = 4): sum_{m = 2..seg} gL^(m - 1)
// local(seg - m), in this order; local(j) sits in segment j + 1's slot.  The
// first term, m = 1, is the item's own phase-A result.
__device__ __forceinline__ void start_sum(const Params &p, int bh, int seg, int r, int g,
                                          float gL, float (&acc)[32]) {
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] = 0.f;
    float w = gL;
    for (int m = 2; m <= seg; ++m) {
        const int pi = item_index(bh, seg - m + 1, p);
        if (!LA_DCHECK(p.status, pi >= 0 && pi < p.items && r >= 0 && r < D)) continue;
        const float *src = p.agg + (size_t)pi * STATE;
        if (g < 4) {
            const float4 *s4 = reinterpret_cast<const float4 *>(src);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float4 x = __ldcg(s4 + (8 * g + u) * 128 + r);
                acc[4 * u] = fmaf(w, x.x, acc[4 * u]);
                acc[4 * u + 1] = fmaf(w, x.y, acc[4 * u + 1]);
                acc[4 * u + 2] = fmaf(w, x.z, acc[4 * u + 2]);
                acc[4 * u + 3] = fmaf(w, x.w, acc[4 * u + 3]);
            }
        } else {
            acc[0] = fmaf(w, __ldcg(src + D * D + r), acc[0]);
        }
        w *= gL;
    }
}

// ---------------------------------------------------------------- producer

// One job per chunk: phase A jobs load K and V (kept in L2 for phase B),
// phase B jobs load K, Q and V.  Phase A's tiles go to L2 kPrefetch jobs
// ahead.  Phase B's are not prefetched: with every SM streaming, prefetched
// lines were evicted before their loads came, and read twice.
// A V slot that a phase-B chunk used holds that chunk's output once the
// output epilogue releases it: the producer writes it out (two TMA stores)
// and waits until they have read the slot before it loads into it again.
__device__ __forceinline__ void store_staged(uint8_t *smem, const CUtensorMap *to, int st,
                                             int c, int bh) {
    tma_store_3d(to, smem + v_off(st), 0, c * C, bh);
    tma_store_3d(to, smem + v_off(st) + v_lbo(st), 64, c * C, bh);
    tma_store_commit();
    tma_store_wait_read<0>();
}

__device__ void producer(uint8_t *smem, Small &sm, const Params &p, const Ctx &cx,
                         const CUtensorMap *tq, const CUtensorMap *tk,
                         const CUtensorMap *tv, const CUtensorMap *to) {
    const uint64_t keep = policy_evict_last(), stream = policy_evict_first();
    int j = 0, jk = 0, nq = 0, tl = 0;
    // per V slot: the output chunk and head staged there (-1: none)
    int out_c[STAGES] = {-1, -1}, out_bh[STAGES] = {0, 0};
    for (;;) {
        int t = atomicAdd(p.ctrl, 1);
        if (t >= p.items || *cx.abort) t = -1;
        const int r = tl & 1;
        settle_wait(&sm.item_empty[r], ((tl >> 1) & 1) ^ 1);
        ((volatile int *)sm.ring)[r] = t;
        mbar_arrive(&sm.item_full[r]);
        ++tl;
        if (t < 0) break;
        const Item it = decode_item(t, p);
        (void)LA_DCHECK(p.status, it.bh >= 0 && it.bh < p.BH && it.seg < p.nseg && it.a0 >= 0 &&
                                      it.a0 <= it.a1 && it.a1 == it.c0 && it.c0 < it.c1 &&
                                      it.c1 <= p.nchunks);
        const int nc = it.c1 - it.c0, nA = it.hasA ? it.a1 - it.a0 : 0, nJ = nA + nc;
        if (*cx.abort) continue;  // issue nothing more once a wait gave up
        bool stop = false;
        for (int x = 0; x < nJ + kPrefetch && !stop; ++x) {
            if (x < nJ) {  // prefetch of job x, then the loads of job x - kPrefetch
                const int pass = x < nA ? 0 : 1;
                const int c = pass == 0 ? it.a0 + x : it.c0 + (x - nA);
                if (pass == 0) {
                    for (int kb = 0; kb < 2; ++kb) {
                        tma_prefetch_3d(tk, 64 * kb, c * C, it.bh, keep);
                        tma_prefetch_3d(tv, 64 * kb, c * C, it.bh, keep);
                    }
                }
            }
            const int y = x - kPrefetch;
            if (y < 0) continue;
            const int pass = y < nA ? 0 : 1;
            const int c = pass == 0 ? it.a0 + y : it.c0 + (y - nA);
            const int st = j % STAGES;
            const uint32_t par = ((j / STAGES) & 1) ^ 1;
            if (!wait_bar_spin(&sm.k_empty[st], par, cx)) break;
            // one arming per phase: the slot's previous load has landed (it
            // always has unless a wait gave up and let a consumer run ahead)
            if (j >= STAGES) settle_wait(&sm.k_full[st], par);
            mbar_arrive_expect_tx(&sm.k_full[st], TILE);
            for (int kb = 0; kb < 2; ++kb)
                tma_load_3d(smem + k_off(st) + kb * BLK, tk, &sm.k_full[st], 64 * kb,
                            c * C, it.bh, pass == 0 ? keep : stream);
            ++jk;
            if (pass == 1) {
                if (!wait_bar_spin(&sm.q_empty, (nq & 1) ^ 1, cx)) break;
                if (nq > 0) settle_wait(&sm.q_full, (nq & 1) ^ 1);
                mbar_arrive_expect_tx(&sm.q_full, TILE);
                for (int kb = 0; kb < 2; ++kb)
                    tma_load_3d(smem + OFF_Q + kb * BLK, tq, &sm.q_full, 64 * kb, c * C,
                                it.bh, stream);
                ++nq;
            }
            if (!wait_bar_spin(&sm.v_empty[st], par, cx)) {
                stop = true;
                break;
            }
            if (out_c[st] >= 0) store_staged(smem, to, st, out_c[st], out_bh[st]);
            out_c[st] = pass == 1 ? c : -1;
            out_bh[st] = it.bh;
            if (j >= STAGES) settle_wait(&sm.v_full[st], par);
            mbar_arrive_expect_tx(&sm.v_full[st], TILE);
            for (int kb = 0; kb < 2; ++kb)
                tma_load_3d(smem + v_off(st) + kb * v_lbo(st), tv, &sm.v_full[st], 64 * kb,
                            c * C, it.bh, pass == 0 ? keep : stream);
            ++j;
        }
    }
    // the outputs still staged (the last phase-B chunks), once released
    for (int x = j - STAGES; x < j; ++x) {
        if (x < 0) continue;
        const int st = x % STAGES;
        if (out_c[st] < 0 || *cx.abort) continue;
        if (wait_bar_spin(&sm.v_empty[st], (x / STAGES) & 1, cx))
            store_staged(smem, to, st, out_c[st], out_bh[st]);
    }
    tma_store_wait_all<0>();
    // the last loads of each slot have landed before the CTA may exit
    for (int x = jk - STAGES; x < jk; ++x)
        if (x >= 0) settle_wait(&sm.k_full[x % STAGES], (x / STAGES) & 1);
    for (int x = j - STAGES; x < j; ++x)
        if (x >= 0) settle_wait(&sm.v_full[x % STAGES], (x / STAGES) & 1);
    if (nq > 0) settle_wait(&sm.q_full, (nq - 1) & 1);
}

// ---------------------------------------------------------------- MMA issuer

template <int kMode>
__device__ void mma_issuer(uint8_t *smem, Small &sm, const Params &p,
                           const Ctx &cx, uint32_t tmem) {
    // P = phi(Q) phi(K)^T: A = phi(Q) (TMEM), B = phi(K) (K-major)
    constexpr uint32_t idP = idesc_bf16(128, 128, 0, 0);
    // Khat^T [V | 1]: A = Khat^T (MN-major: features contiguous), B MN-major
    constexpr uint32_t idSU = idesc_bf16(128, NX, 1, 1);
    // Qhat [S | z]: A = Qhat (TMEM), B = bf16 [S | z] (MN-major)
    constexpr uint32_t idQS = idesc_bf16(128, NX, 0, 1);
    // Pt [V | 1]: A = Pt (TMEM), B MN-major
    constexpr uint32_t idPV = idesc_bf16(128, NX, 0, 1);
    const uint32_t sb = smem_u32(smem + OFF_SB);
    int j = 0, nb = 0, nsb = 0, tl = 0;
    for (;;) {
        const int t = pop_item(sm, tl, cx, 0, 0, true);
        if (t < 0) break;
        const Item it = decode_item(t, p);
        if (it.hasA) {
            // phase A: the predecessor's local state Khat^T [V | 1] into S | z
            for (int c = it.a0; c < it.a1; ++c, ++j) {
                const int st = j % STAGES;
                wait_bar_spin(&sm.xfk[st], (j / STAGES) & 1, cx);
                wait_bar_spin(&sm.v_full[st], (j / STAGES) & 1, cx);
                tc_fence_after();
                const uint32_t kb = smem_u32(smem + k_off(st));
                const uint32_t vb = smem_u32(smem + v_off(st));
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    mma_ss(tmem + TM_S, sdesc_sw128(kb + ks * 2048, BLK, 1024),
                           sdesc_sw128(vb + ks * 2048, v_lbo(st), 1024), idSU,
                           (c > it.a0 || ks > 0) ? 1u : 0u);
                if (c == it.a1 - 1) mma_commit(&sm.s_full);
                mma_commit(&sm.k_empty[st]);
                mma_commit(&sm.v_empty[st]);
            }
        }
        // phase B.  The state after the item's last chunk is only needed as
        // the sequence's final state; otherwise that chunk has no update.
        const int nB = it.c1 - it.c0;
        const bool final_state = p.S_out && it.seg == p.nseg - 1;
        for (int qi = 0; qi < nB; ++qi, ++j, ++nb) {
            const int st = j % STAGES;
            const uint32_t sp = (j / STAGES) & 1, cp = nb & 1;
            const bool su = qi + 1 < nB || final_state;
            const uint32_t kb = smem_u32(smem + k_off(st));
            const uint32_t vb = smem_u32(smem + v_off(st));
            // P once phi(K), phi(Q) are in place and the previous Pt [V | 1]
            // has released the P columns
            wait_bar_spin(&sm.xfk[st], sp, cx);
            wait_bar_spin(&sm.xfq, cp, cx);
            wait_bar_spin(&sm.pv_done, cp ^ 1, cx);
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_ts(tmem + TM_P, tmem + TM_Q + ks * 8,
                       sdesc_sw128(kb + kmajor_off(ks, BLK), 16, 1024), idP,
                       ks > 0 ? 1u : 0u);
            mma_commit(&sm.pfull);
            // the state before this chunk (TMEM S | z pre-scaled by g^n and
            // its bf16 copy); with decay Khat, Qhat weighted in place
            wait_bar_spin(&sm.sb_ready, nsb & 1, cx);
            ++nsb;
            if (kMode == 1) wait_bar_spin(&sm.khat_ready, cp, cx);
            wait_bar_spin(&sm.v_full[st], sp, cx);
            tc_fence_after();
            if (su) {
#pragma unroll
                for (int ks = 0; ks < C / 16; ++ks)
                    mma_ss(tmem + TM_S, sdesc_sw128(kb + ks * 2048, BLK, 1024),
                           sdesc_sw128(vb + ks * 2048, v_lbo(st), 1024), idSU, 1u);
            }
            mma_commit(&sm.k_empty[st]);
            // O is free once the output epilogue has read the previous chunk's
            wait_bar_spin(&sm.o_empty, cp ^ 1, cx);
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_ts(tmem + TM_O, tmem + TM_Q + ks * 8,
                       sdesc_sw128(sb + ks * 2048, BLK, 1024), idQS, ks > 0 ? 1u : 0u);
            // the state warps may now read S | z and rewrite [S | z]; the
            // feature map may write the next chunk's phi(Q)
            mma_commit(&sm.s_full);
            mma_commit(&sm.q_free);
            wait_bar_spin(&sm.pt_ready, cp, cx);
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < C / 16; ++ks)
                mma_ts(tmem + TM_O, tmem + TM_P + ks * 8,
                       sdesc_sw128(vb + ks * 2048, v_lbo(st), 1024), idPV, 1u);
            mma_commit(&sm.o_full);
            mma_commit(&sm.pv_done);
        }
        if (final_state) {
            // S's columns are reused by the next item: wait until the state
            // warps have written the final state out
            wait_bar_spin(&sm.sb_ready, nsb & 1, cx);
            ++nsb;
        }
    }
    // every product has completed before TMEM is released
    mma_commit(&sm.fin);
    settle_wait(&sm.fin, 0);
}

// ---------------------------------------------------------------- transform

// phi on this thread's 64 features (part) of row `row` of the Q landing
// tile, packed bf16 pairs in feature order (the A operand's TMEM layout).
__device__ __forceinline__ void phi_q_row(const uint8_t *tile, int row, int part,
                                          bool phi, uint32_t (&w)[32]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 x = *reinterpret_cast<const uint4 *>(
            tile + part * BLK + sw128_offset(row, i * 8));
        w[4 * i] = phi ? phi2(x.x) : x.x;
        w[4 * i + 1] = phi ? phi2(x.y) : x.y;
        w[4 * i + 2] = phi ? phi2(x.z) : x.z;
        w[4 * i + 3] = phi ? phi2(x.w) : x.w;
    }
}

// phi(K) times w on this thread's half of a K row, in place; one copy of
// the code for every call site (the feature map's warps share their
// instruction cache with the MMA issuer and the epilogues).  w = 1 leaves
// phi(K) exact; w = 0 zeroes the rows past the sequence end.
static __device__ __noinline__ void feature_k_row(uint8_t *kt, int row, int part,
                                                  uint32_t w2, bool phi) {
    transform_row_scaled<D>(kt, row, part, w2, phi);
}

template <int kMode>
__device__ void transform(uint8_t *smem, Small &sm, const Params &p,
                          const Ctx &cx, const DecayArgs &dk, uint32_t tmem) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int et = threadIdx.x - kWarpT * 32;  // 0..255
    // row = the TMEM lane this warp may access; part = half of the features
    const int row = 32 * (warp & 3) + lane, part = (warp - kWarpT) >> 2;
    const uint32_t lq = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + TM_Q + 32 * part;
    int j = 0, nb = 0, tl = 0;
    for (;;) {
        const int t = pop_item(sm, tl, cx, BAR_T, kTThreads, et == 0);
        if (t < 0) break;
        const Item it = decode_item(t, p);
        const float lg = head_log2g(dk, it.bh);
        if (it.hasA) {
            // phase A over the predecessor's chunks [a0, a1): Khat_t =
            // g^(a1 C - 1 - t) phi(k_t), t relative to the item's own start
            // (every chunk of the range is full)
            const int seg_end = it.a1 * C;
            for (int c = it.a0; c < it.a1; ++c, ++j) {
                const int st = j % STAGES;
                wait_bar(&sm.k_full[st], (j / STAGES) & 1, cx);
                uint8_t *kt = smem + k_off(st);
                const int tok = c * C + row;
                if (kMode || tok >= p.N) {
                    const float w = tok < p.N ? gpow(lg, seg_end - 1 - tok) : 0.f;
                    feature_k_row(kt, row, part, bf2_splat(w), p.phi != 0);
                } else {
                    feature_k_row(kt, row, part, kBf16One2, p.phi != 0);
                }
                fence_async_shared();
                named_bar_sync(BAR_T, kTThreads);
                if (et == 0) mbar_arrive(&sm.xfk[st]);
            }
        }
        for (int c = it.c0; c < it.c1; ++c, ++j, ++nb) {
            const int st = j % STAGES;
            const int n = min(C, p.N - c * C);
            uint8_t *kt = smem + k_off(st);
            wait_bar(&sm.k_full[st], (j / STAGES) & 1, cx);
            if (kMode == 2) {  // Khat_t = g^(n-1-t) phi(k_t) at once (rows past N -> 0)
                const float wk = row >= n ? 0.f : gpow(lg, n - 1 - row);
                feature_k_row(kt, row, part, bf2_splat(wk), p.phi != 0);
            } else {
                // rows past N -> 0
                feature_k_row(kt, row, part, row >= n ? 0u : kBf16One2, p.phi != 0);
            }
            fence_async_shared();
            named_bar_sync(BAR_T, kTThreads);
            if (et == 0) mbar_arrive(&sm.xfk[st]);
            // phi(Q) from the landing slot into TMEM, once the previous
            // chunk's last product has read phi(Q)'s columns
            wait_bar(&sm.q_full, nb & 1, cx);
            uint32_t w[32];
            phi_q_row(smem + OFF_Q, row, part, p.phi != 0, w);
            if (kMode == 2) {  // Q'_i = g^(i+1-n) phi(q_i) at once
                const uint32_t wq = bf2_splat(gpow(lg, row + 1 - n));
#pragma unroll
                for (int e = 0; e < 32; ++e) w[e] = bf2_mul(w[e], wq);
            }
            named_bar_sync(BAR_T, kTThreads);
            if (et == 0) mbar_arrive(&sm.q_empty);
            wait_bar(&sm.q_free, (nb & 1) ^ 1, cx);
            tc_fence_after();
            tmem_st32(lq, w);
            tmem_wait_st();
            tc_fence_before();
            named_bar_sync(BAR_T, kTThreads);
            if (et == 0) mbar_arrive(&sm.xfq);
            if (kMode == 1) {
                // once P(c) has read the unweighted rows: Khat_t =
                // g^(n-1-t) phi(k_t) in place, Qhat_i = g^(i+1) phi(q_i) in TMEM
                wait_bar(&sm.pfull, nb & 1, cx);
                tc_fence_after();
                const float wk = row >= n ? 0.f : gpow(lg, n - 1 - row);
                const uint32_t wq = bf2_splat(gpow(lg, row + 1));
                scale_row<D>(kt, row, part, bf2_splat(wk));
#pragma unroll
                for (int e = 0; e < 32; ++e) w[e] = bf2_mul(w[e], wq);
                tmem_st32(lq, w);
                tmem_wait_st();
                fence_async_shared();
                tc_fence_before();
                named_bar_sync(BAR_T, kTThreads);
                if (et == 0) mbar_arrive(&sm.khat_ready);
            }
        }
    }
}

// ---------------------------------------------------------------- score + output

// Causal mask and decay on P (fp32, TMEM), rounded to bf16 in place (the A
// operand of Pt [V | 1]).  One thread per row (= TMEM lane).  With the
// weights folded into both operands (mode 2) P already holds
// g^(i - j) phi(q_i) . phi(k_j): only the mask remains.
template <int kMode>
__device__ __forceinline__ void score_chunk(Small &sm, const Ctx &cx, uint32_t lb,
                                            int q, int lane, float lg, int nb) {
    const uint32_t tp = lb + TM_P;
    const int row = q * 32 + lane;
    wait_bar(&sm.pfull, nb & 1, cx);
    tc_fence_after();
#pragma unroll 1
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
                if (kMode == 1) {
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
                    if (e <= lane) x0 = kMode == 1 ? u2f(v[e]) * sm.gtab[lane - e] : u2f(v[e]);
                    if (e + 1 <= lane)
                        x1 = kMode == 1 ? u2f(v[e + 1]) * sm.gtab[lane - e - 1] : u2f(v[e + 1]);
                    pk[e >> 1] = pack_bf16x2(x0, x1);
                }
            }
        }
        tmem_st16(tp + 16 * blk, pk);
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&sm.pt_ready);  // 128 arrivals, one per row
}

// One chunk's output: O / den (O alone without the normaliser) in bf16,
// staged into the chunk's V slot (V is dead once Pt [V | 1] has completed).
// O is released as soon as it has been read; the staged tile is handed to
// the producer (v_empty), which writes it out with two TMA stores before it
// loads the next V into the slot.
__device__ __forceinline__ void output_chunk(uint8_t *smem, Small &sm, const Ctx &cx,
                                             uint32_t lb, int row, int et, int nb, int st,
                                             bool norm) {
    wait_bar(&sm.o_full, nb & 1, cx);
    tc_fence_after();
    float inv = 1.f;
    if (norm) {
        uint32_t dr = tmem_ld1(lb + TM_O + D);
        tmem_wait_ld();
        reg_fence(dr);
        inv = 1.f / u2f(dr);
    }
    uint8_t *vs = smem + v_off(st);
#pragma unroll 1
    for (int g = 0; g < 4; ++g) {
        uint32_t o[32];
        tmem_ld32(lb + TM_O + 32 * g, o);
        tmem_wait_ld();
        reg_fence(o);
        if (g == 3) {
            tc_fence_before();
            mbar_arrive(&sm.o_empty);  // 128 arrivals: O has been read
        }
        uint8_t *blk = vs + (g >> 1) * v_lbo(st);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
            *reinterpret_cast<uint4 *>(blk + sw128_offset(row, 32 * (g & 1) + 8 * ch)) =
                make_uint4(pack_bf16x2(u2f(o[8 * ch]) * inv, u2f(o[8 * ch + 1]) * inv),
                           pack_bf16x2(u2f(o[8 * ch + 2]) * inv, u2f(o[8 * ch + 3]) * inv),
                           pack_bf16x2(u2f(o[8 * ch + 4]) * inv, u2f(o[8 * ch + 5]) * inv),
                           pack_bf16x2(u2f(o[8 * ch + 6]) * inv, u2f(o[8 * ch + 7]) * inv));
    }
    fence_async_shared();
    named_bar_sync(BAR_E1, 128);
    if (et == 0) mbar_arrive(&sm.v_empty[st]);
}

template <int kMode>
__device__ void score_output(uint8_t *smem, Small &sm, const Params &p, const Ctx &cx,
                             const DecayArgs &dk, uint32_t tmem) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3, row = q * 32 + lane;
    const int et = threadIdx.x - kWarpE1 * 32;
    const uint32_t lb = tmem + ((uint32_t)(q * 32) << 16);
    const bool norm = p.norm != 0;
    int nb = 0, j = 0, tl = 0;
    for (;;) {
        const int t = pop_item(sm, tl, cx, BAR_E1, 128, et == 0);
        if (t < 0) break;
        const Item it = decode_item(t, p);
        const float lg = head_log2g(dk, it.bh);
        if (kMode == 1 && et < 32) sm.gtab[et] = gpow(lg, et);
        // The published part of the start state (segments 1 .. seg-1), if
        // they have all published already, summed now (phase A runs
        // meanwhile) into TMEM O (row `row` of S, and z in column D); the
        // state warps take it from there.
        if (et < 32) {
            const bool e = it.seg >= 2 && preds_published(p, cx, it.bh, it.seg, lane, false);
            if (lane == 0) sm.lb_early = e ? 1 : 0;
        }
        named_bar_sync(BAR_E1, 128);
        if (sm.lb_early) {
            const float gL = gpow(lg, p.seg_chunks * C);
#pragma unroll 1
            for (int g = 0; g < 5; ++g) {
                float acc[32];
                start_sum(p, it.bh, it.seg, row, g, gL, acc);
                if (g < 4) {
                    uint32_t w[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(acc[e]);
                    tmem_st32(lb + TM_O + 32 * g, w);
                } else {
                    uint32_t zw[16];
                    zw[0] = __float_as_uint(acc[0]);
#pragma unroll
                    for (int e = 1; e < 16; ++e) zw[e] = 0u;
                    tmem_st16(lb + TM_O + D, zw);
                }
            }
            tmem_wait_st();
        }
        tc_fence_before();
        named_bar_sync(BAR_E1, 128);
        if (et == 0) mbar_arrive(&sm.lb_done);
        // phase B: the output of chunk c - 1 (its O completes before P of
        // chunk c, issued after it), then the scores of chunk c
        if (it.hasA) j += it.a1 - it.a0;
        for (int c = it.c0; c < it.c1; ++c, ++nb, ++j) {
            if (c > it.c0)
                output_chunk(smem, sm, cx, lb, row, et, nb - 1, (j - 1) % STAGES, norm);
            score_chunk<kMode>(sm, cx, lb, q, lane, lg, nb);
        }
        output_chunk(smem, sm, cx, lb, row, et, nb - 1, (j - 1) % STAGES, norm);
    }
}

// ---------------------------------------------------------------- state

// 32 values of row a, columns [32 g, 32 g + 32), into the bf16 [S | z]
// operand (S blocks 0 and 1).
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

// z[a] in bf16 at column 0 of the z block of [S | z].
__device__ __forceinline__ void store_zb(uint8_t *sb, int a, float z) {
    *reinterpret_cast<__nv_bfloat16 *>(sb + 2 * BLK + sw128_offset(a, 0)) =
        __float2bfloat16_rn(z);
}

// The z column of the S | z accumulator: (z, 0, ..., 0) over 16 columns.
__device__ __forceinline__ void tmem_put_z(uint32_t taddr, float z) {
    uint32_t v[16];
    v[0] = __float_as_uint(z);
#pragma unroll
    for (int e = 1; e < 16; ++e) v[e] = 0u;
    tmem_st16(taddr, v);
}

template <int kMode>
__device__ void state_role(uint8_t *smem, Small &sm, const Params &p, const Ctx &cx,
                           const DecayArgs &dk, uint32_t tmem) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;
    const int et = threadIdx.x - kWarpE2 * 32;
    const int a = q * 32 + lane;  // TMEM lane = state row (key feature)
    const uint32_t lb = tmem + ((uint32_t)(q * 32) << 16);
    uint8_t *sb = smem + OFF_SB;
    int ns = 0, nl = 0, tl = 0;
    for (;;) {
        const int t = pop_item(sm, tl, cx, BAR_E2, 128, et == 0);
        if (t < 0) break;
        const Item it = decode_item(t, p);
        const float lg = head_log2g(dk, it.bh);
        const float gL = gpow(lg, p.seg_chunks * C);
        const float f0 = gpow(lg, min(C, p.N - it.c0 * C));
        if (it.hasA) {
            // phase A done: its result (the predecessor's local state) is in
            // TMEM S; publish it at once if a later segment needs it
            wait_bar(&sm.s_full, ns & 1, cx);
            ++ns;
            tc_fence_after();
            if (it.pub) {
                // (a debug check guards the stores only: every thread still
                // reaches the barrier)
                const bool okp = LA_DCHECK(p.status, t < p.items && a < D);
                float4 *d4 = reinterpret_cast<float4 *>(p.agg + (size_t)t * STATE);
#pragma unroll 1
                for (int g = 0; g < 4; ++g) {
                    uint32_t v[32];
                    tmem_ld32(lb + TM_S + 32 * g, v);
                    tmem_wait_ld();
                    reg_fence(v);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        if (okp)
                            d4[(8 * g + u) * 128 + a] =
                                make_float4(u2f(v[4 * u]), u2f(v[4 * u + 1]),
                                            u2f(v[4 * u + 2]), u2f(v[4 * u + 3]));
                }
                uint32_t zl = tmem_ld1(lb + TM_S + D);
                tmem_wait_ld();
                reg_fence(zl);
                if (okp) p.agg[(size_t)t * STATE + D * D + a] = u2f(zl);
                __threadfence();
                named_bar_sync(BAR_E2, 128);
                if (et == 0 && it.seg != p.hold_seg && okp) publish_flag(p.flags + t, FLAG_AGG);
            }
        }
        // The start state: the own phase-A result (TMEM S) plus the part
        // that segments 1 .. seg-1 published, summed by the score warps
        // during phase A (parked in TMEM O), or here once they have all
        // published.
        wait_bar(&sm.lb_done, nl & 1, cx);
        ++nl;
        tc_fence_after();
        const bool lbk = it.seg >= 2;
        // one value per warp; the barrier below is passed whatever it is, so
        // that the role's barrier count follows from the item alone
        const bool early = __shfl_sync(~0u, sm.lb_early, 0) != 0;
        if (lbk && !early && warp == kWarpE2)
            preds_published(p, cx, it.bh, it.seg, lane, true);
        named_bar_sync(BAR_E2, 128);
#pragma unroll 1
        for (int g = 0; g < 5; ++g) {
            // g = 4: the z column
            float pv[32];
            if (!lbk) {
#pragma unroll
                for (int e = 0; e < 32; ++e) pv[e] = 0.f;
            } else if (early) {
                if (g < 4) {
                    uint32_t v[32];
                    tmem_ld32(lb + TM_O + 32 * g, v);
                    tmem_wait_ld();
                    reg_fence(v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) pv[e] = u2f(v[e]);
                } else {
                    uint32_t zr = tmem_ld1(lb + TM_O + D);
                    tmem_wait_ld();
                    reg_fence(zr);
                    pv[0] = u2f(zr);
                }
            } else {
                start_sum(p, it.bh, it.seg, a, g, gL, pv);
            }
            if (it.hasA) {  // + the own phase-A result, the first term
                if (g < 4) {
                    uint32_t v[32];
                    tmem_ld32(lb + TM_S + 32 * g, v);
                    tmem_wait_ld();
                    reg_fence(v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) pv[e] = u2f(v[e]) + pv[e];
                } else {
                    uint32_t zl = tmem_ld1(lb + TM_S + D);
                    tmem_wait_ld();
                    reg_fence(zl);
                    pv[0] = u2f(zl) + pv[0];
                }
            }
            if (g == 4) {
                store_zb(sb, a, kMode == 2 ? f0 * pv[0] : pv[0]);
                tmem_put_z(lb + TM_S + D, f0 * pv[0]);
                continue;
            }
            if (kMode == 2) {  // the operand carries g^n (see the feature map)
                float ps[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) ps[e] = f0 * pv[e];
                store_sb32(sb, a, g, ps);
            } else {
                store_sb32(sb, a, g, pv);
            }
            // phase-B start: TMEM S = g^n0 S_start
            uint32_t w[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) w[e] = __float_as_uint(f0 * pv[e]);
            tmem_st32(lb + TM_S + 32 * g, w);
        }
        tmem_wait_st();
        fence_async_shared();
        tc_fence_before();
        named_bar_sync(BAR_E2, 128);
        if (et == 0) mbar_arrive(&sm.sb_ready);
        // phase B: per chunk, once its Khat^T [V | 1] and Qhat [S | z] have
        // completed, the bf16 [S | z] of the next chunk and with decay the
        // rescale g^n of the accumulator
        for (int c = it.c0; c < it.c1; ++c) {
            wait_bar(&sm.s_full, ns & 1, cx);
            ++ns;
            tc_fence_after();
            if (c + 1 < it.c1) {
                const float f = gpow(lg, min(C, p.N - (c + 1) * C));
#pragma unroll 1
                for (int g = 0; g < 4; ++g) {
                    uint32_t v[32];
                    tmem_ld32(lb + TM_S + 32 * g, v);
                    tmem_wait_ld();
                    reg_fence(v);
                    float x[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[e] = kMode == 2 ? f * u2f(v[e]) : u2f(v[e]);
                    store_sb32(sb, a, g, x);
                    if (kMode == 1) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(f * x[e]);
                    } else if (kMode == 2) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(x[e]);
                    }
                    if (kMode) tmem_st32(lb + TM_S + 32 * g, v);
                }
                uint32_t zr = tmem_ld1(lb + TM_S + D);
                tmem_wait_ld();
                reg_fence(zr);
                store_zb(sb, a, kMode == 2 ? f * u2f(zr) : u2f(zr));
                if (kMode) {
                    tmem_put_z(lb + TM_S + D, f * u2f(zr));
                    tmem_wait_st();
                }
                fence_async_shared();
                tc_fence_before();
                named_bar_sync(BAR_E2, 128);
                if (et == 0) mbar_arrive(&sm.sb_ready);
            }
        }
        if (p.S_out && it.seg == p.nseg - 1) {
            const bool oks = LA_DCHECK(p.status, it.bh < p.BH && a < D);
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
                    if (oks)
                        d4[u] = make_float4(u2f(v[4 * u]), u2f(v[4 * u + 1]), u2f(v[4 * u + 2]),
                                            u2f(v[4 * u + 3]));
            }
            uint32_t zr = tmem_ld1(lb + TM_S + D);
            tmem_wait_ld();
            reg_fence(zr);
            if (oks) p.z_out[(size_t)it.bh * D + a] = u2f(zr);
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
                   const __grid_constant__ CUtensorMap tv,
                   const __grid_constant__ CUtensorMap to, const Params p,
                   const DecayArgs dk) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    Small &sm = *reinterpret_cast<Small *>(smem + OFF_SMALL);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Ctx cx{reinterpret_cast<volatile int *>(p.ctrl + 1), p.status, p.timeout};
    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, 1);
        mbar_init(&sm.q_empty, 1);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&sm.k_full[s], 1);
            mbar_init(&sm.k_empty[s], 1);
            mbar_init(&sm.v_full[s], 1);
            mbar_init(&sm.v_empty[s], 1);
            mbar_init(&sm.xfk[s], 1);
        }
        mbar_init(&sm.xfq, 1);
        mbar_init(&sm.q_free, 1);
        mbar_init(&sm.khat_ready, 1);
        mbar_init(&sm.pfull, 1);
        mbar_init(&sm.pt_ready, 128);
        mbar_init(&sm.pv_done, 1);
        mbar_init(&sm.o_full, 1);
        mbar_init(&sm.o_empty, 128);
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.sb_ready, 1);
        mbar_init(&sm.lb_done, 1);
        for (int r = 0; r < 2; ++r) {
            mbar_init(&sm.item_full[r], 1);
            mbar_init(&sm.item_empty[r], 4);
        }
        mbar_init(&sm.fin, 1);
        fence_mbar_init();
    }
    // constant operand blocks: the ones block of [V | 1] (column 0 is one)
    // and the z block of [S | z] (column 0 rewritten per chunk, rest zero)
    for (int i = threadIdx.x; i < BLK / 16; i += kThreads) {
        reinterpret_cast<uint4 *>(smem + OFF_ONES)[i] = make_uint4(0u, 0u, 0u, 0u);
        reinterpret_cast<uint4 *>(smem + OFF_SB + 2 * BLK)[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();
    if (threadIdx.x < C)
        *reinterpret_cast<uint16_t *>(smem + OFF_ONES + sw128_offset(threadIdx.x, 0)) =
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
        if (lane == 0) producer(smem, sm, p, cx, &tq, &tk, &tv, &to);
    } else if (warp == 1) {
        if (lane == 0) mma_issuer<kMode>(smem, sm, p, cx, tmem);
    } else if (warp < kWarpE1) {
        transform<kMode>(smem, sm, p, cx, dk, tmem);
    } else if (warp < kWarpE2) {
        score_output<kMode>(smem, sm, p, cx, dk, tmem);
    } else {
        state_role<kMode>(smem, sm, p, cx, dk, tmem);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TM_COLS);
}

constexpr size_t kSmemBytes = (size_t)OFF_SMALL + sizeof(Small) + 1024;
static_assert(kSmemBytes <= 232448, "shared memory budget");
static_assert(OFF_Q % 1024 == 0 && OFF_K0 % 1024 == 0 && OFF_K1 % 1024 == 0 &&
                  OFF_V0 % 1024 == 0 && OFF_V1 % 1024 == 0 && OFF_ONES % 1024 == 0,
              "SW128 tiles need 1024-byte alignment");
static_assert(TM_Q + 64 <= TM_COLS, "TMEM columns");

}  // namespace causal_wide

namespace {

inline size_t align_up_w(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Work decomposition and workspace layout of one launch.
struct WidePlan {
    int seg_chunks, seg0, nseg, nchunks;
    long long items;
    size_t off_flags, off_agg, total;
};

WidePlan plan_wide(const FwdShape &sh, int seg_chunks, int sms) {
    using namespace causal_wide;
    WidePlan pl{};
    pl.nchunks = (sh.N + C - 1) / C;
    const bool automatic = seg_chunks <= 0;
    if (automatic) seg_chunks = wide_segment_chunks(sh.BH(), pl.nchunks, sms);
    if (seg_chunks > pl.nchunks) seg_chunks = pl.nchunks;
    int seg0 = seg_chunks;
    // Two segments per head: segment 0 runs phase B from the start while
    // segment 1 first reduces segment 0's chunks, so segment 0 takes three
    // fifths of them.
    if (automatic && (pl.nchunks + seg_chunks - 1) / seg_chunks == 2) {
        seg0 = 3 * pl.nchunks / 5;
        seg_chunks = pl.nchunks - seg0;
    }
    pl.seg0 = seg0;
    pl.seg_chunks = seg_chunks;
    pl.nseg = pl.nchunks <= seg0 ? 1 : 1 + (pl.nchunks - seg0 + seg_chunks - 1) / seg_chunks;
    pl.items = sh.BH() * pl.nseg;
    pl.off_flags = 256;
    pl.off_agg = align_up_w(pl.off_flags + sizeof(int) * (size_t)pl.items, 256);
    pl.total = pl.off_agg +
               (pl.nseg > 1 ? sizeof(float) * (size_t)STATE * (size_t)pl.items : 0);
    return pl;
}

TcResult launch_wide_with(const void *q, const void *k, const void *v, void *out,
                          const FwdShape &sh, const DecayArgs &dk, const WidePlan &pl,
                          int *status, char *ws, float *S_out, float *z_out,
                          cudaStream_t stream, int sms) {
    using namespace causal_wide;
    const int BH = (int)sh.BH(), N = sh.N;
    CUtensorMap tq, tk, tv, to;
    cudaError_t e;
    if ((e = tchost::make_seq_map(&tq, q, BH, N, D, C)) != cudaSuccess ||
        (e = tchost::make_seq_map(&tk, k, BH, N, D, C)) != cudaSuccess ||
        (e = tchost::make_seq_map(&tv, v, BH, N, D, C)) != cudaSuccess ||
        (e = tchost::make_seq_map(&to, out, BH, N, D, C)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward: TMA descriptor"};
    Params p{};
    p.BH = BH;
    p.N = N;
    p.nchunks = pl.nchunks;
    p.seg_chunks = pl.seg_chunks;
    p.seg0 = pl.seg0;
    p.nseg = pl.nseg;
    p.items = (int)pl.items;
    p.timeout = 1LL << 32;
    p.hold_seg = -1;
    tc_debug_take_timeout(&p.timeout, &p.hold_seg);
    p.S_out = S_out;
    p.z_out = z_out;
    p.phi = sh.phi;
    p.norm = sh.norm;
    p.ctrl = reinterpret_cast<int *>(ws);
    p.flags = reinterpret_cast<int *>(ws + pl.off_flags);
    p.agg = reinterpret_cast<float *>(ws + pl.off_agg);
    p.status = status;
    // the ticket counter, abort flag and segment flags start at zero; the
    // published states need no clearing
    if ((e = tc_zero_words(ws, pl.off_agg, stream)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward: workspace clear"};
    // With every decay at least kFoldMin the weights fold into both operands
    // (mode 2): the largest power in P, g^(2C - 1), stays above 2^-96 and
    // g^-C below 2^49.  Only with the elu + 1 map: its positive features keep
    // the rounding of the weighted rows at a relative 2^-8 of P, where the
    // identity map's cancelling terms would not.
    bool fold = dk.has != 0 && sh.phi != 0;
    for (int h = 0; fold && h < dk.H; ++h) fold = dk.g[h] >= kFoldMin;
    auto kern = !dk.has ? causal_wide_kernel<0>
                        : (fold ? causal_wide_kernel<2> : causal_wide_kernel<1>);
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kSmemBytes)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward: kernel attribute"};
    const int grid = (int)(pl.items < sms ? pl.items : sms);
    e = tchost::launch_dependent(kern, (unsigned)grid, kThreads, kSmemBytes, stream, tq, tk, tv,
                                 to, p, dk);
    if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward: causal kernel launch"};
    note_launches(2);  // workspace clear + forward
    return {LA_OK, cudaSuccess, ""};
}

}  // namespace

// Segment length for the d = 128 kernel: as many segments per head as let
// all items run in one wave (one item per SM), at most 16 (a segment's
// look-back reads every predecessor's local state).  Measured on the
// long-context and decay workloads, one wave of long segments beats several
// waves of short ones, whose per-item costs (look-back, publication,
// pipeline fill and drain) outweigh the L2 hits of phase B's re-read of K
// and V.
int wide_segment_chunks(long long heads, int nchunks, int sms) {
    constexpr long long kMaxSegments = 16;
    if (sms < 1) sms = 1;
    long long nseg = heads > 0 ? sms / heads : 1;
    if (nseg < 1) nseg = 1;
    if (nseg > kMaxSegments) nseg = kMaxSegments;
    if (nseg > nchunks) nseg = nchunks;
    return (int)((nchunks + nseg - 1) / nseg);
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
    } else if ((e = tc_workspace_alloc(&ws, pl.total, stream)) != cudaSuccess) {
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
