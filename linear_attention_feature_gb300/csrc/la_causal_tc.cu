// Chunkwise causal linear attention on tcgen05 tensor cores (bf16 in, fp32
// accumulate), with optional per-head decay g.
//
// The method ("Linear Attention", chunkwise parallel form; "Story of
// Attention - Part 5", section 6 block formulas, with the normaliser carried
// like the numerator): the sequence is cut into chunks of C = 128 tokens.
// For a chunk with local rows i, j (0-based) and S, z the state before it:
//   P      = phi(Q) phi(K)^T                       (tcgen05, TMEM fp32)
//   Pt_ij  = P_ij g^(i-j) for j <= i, else 0       (epilogue, rounded bf16)
//   O      = Pt V + diag(g^(i+1)) phi(Q) S         (tcgen05; Pt read from TMEM)
//   den    = Pt 1 + diag(g^(i+1)) phi(Q) z
//   out_i  = O_i / den_i
//   S     <- g^n S + Khat^T V,  Khat_t = g^(n-1-t) phi(k_t)   (n = chunk length)
//   z     <- g^n z + Khat^T 1
// A tcgen05.mma costs about the same for any N up to 128, so the normaliser
// rides along as a 65th column of the wide products: phi(Q) [S | z],
// Pt [V | 1] and Khat^T [V | 1] are single N = 80 MMAs (the extra 64-column
// operand block holds z or ones in its first column).  With decay the K rows
// are rescaled into Khat in place once P has read them.  S and z
// are carried in TMEM in fp32 and copied to shared memory in bf16 as the B
// operand of the next chunk's phi(Q) [S | z], so numerator and denominator
// are formed from the same bf16 operands.  The feature
// map is evaluated on packed bf16 pairs: phi(x) = max(x, 0) + 2^(min(x, 0)
// log2 e), which is elu(x) + 1 with alpha = 1.
//
// This kernel serves d = 64 (all modes) and the gated mode at d = 128; the
// other d = 128 modes run in la_causal_wide.cu.
//
// Sequence parallelism inside a head: a head's chunks are cut into segments
// (segment 0 of `seg0` chunks, the others of `seg_chunks`), and the value
// dimension into halves of 64 columns (d = 128 gives two halves, each with
// all 128 key features).  A work item is (head, segment, half); persistent
// CTAs take items from a ticket counter (so a CTA only ever waits on items
// held by running CTAs).  Segment 0 starts from the zero state and runs the
// chunk loop (phase B) at once.  A later segment s first reduces its
// predecessor's chunks to that segment's local decayed state (phase A:
// Khat^T [V | 1] only, Khat_t = g^(L-1-t) phi(k_t) relative to the end of
// that range, which is its own start); it keeps that state in TMEM as the
// first term of its start state and publishes it when a later segment
// needs it.  The other terms are the states published by segments
// 1 .. s-1 (the local states of segments s-2 .. 0), decayed and added
// nearest first -- a fixed order, so repeated calls are bit-identical.
// A segment's phase B and its successor's phase A read the same K and V
// tiles from the start of the launch, so the later read often finds them in
// L2 (phase A loads them with evict-last).
//
// Warp roles (576 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2-9 feature-map transform, warps 10-13 score epilogue (mask,
// decay, bf16 P~ in TMEM), warps 14-17 state and output epilogue (bf16
// [S | z] operand, look-back; O / den stored from registers).  P and O
// have two TMEM buffers, and the MMA issuer issues P of chunk j+1 ahead of
// P~V of chunk j when it is ready, so the tensor pipe can run
// ... SU(j) P(j+1) P~V(j) QS(j+1) SU(j+1) ... without waiting for an
// epilogue to drain a buffer.  All waits
// are bounded; a wait that runs out sets the device status word to
// LA_ERR_TIMEOUT and an abort flag, after which every wait passes through so
// that the kernel finishes (with invalid output) instead of hanging.
#include "la_tc.h"
#include "la_tc_host.h"
#include "la_tc_common.cuh"
#include "la_tc_ptx.cuh"

#include <cstdio>
#include <mutex>

namespace la {
namespace causal_tc {

using namespace la::tc;
using namespace la::tcc;

constexpr int C = 128;           // chunk length (tokens) = MMA M
constexpr int DV = 64;           // value columns per work item
constexpr int kGateSlotBytes = 2048;  // a chunk's gate slot (mode 2)
constexpr int kWarpT = 2, kNumT = 8, kWarpE1 = 10, kWarpE2 = 14;
constexpr int kThreads = (kWarpE2 + 4) * 32;  // 576
constexpr int kTThreads = kNumT * 32;
constexpr int BAR_T = 1, BAR_E1 = 2, BAR_E2 = 3;
// TMEM columns: P in two buffers (2 x 128); O | den (80) in two buffers;
// S | z (80).  496 of 512 columns.
constexpr uint32_t TM_P = 0, TM_O = 256, TM_S = 416;
constexpr uint32_t TM_COLS = 512;
constexpr int NX = DV + 16;  // extended N of the wide products
// Kernel mode: 0 no decay, 1 per-head decay g, 2 data-dependent gate per
// token.  Modes 1 and 2 share the structure of the weighted kernel (Q and K
// rows weighted in place once P has read them); they differ only in how the
// weights are formed (powers of g, or products of gates).

struct Params {
    int BH, H, N, nchunks, seg_chunks, nseg, nhalf, items;
    int seg0;           // chunks of segment 0 (later segments: seg_chunks)
    float *agg;         // [items][DK * DV + DK]: S rows (a-major), then z
    int *flags;         // [items]
    float *S_out, *z_out;  // final state [BH][DK][DK] / [BH][DK], or NULL
    int phi, norm;         // elu(x) + 1 on q, k (else identity); divide by den
    const float *gates;    // mode 2: alpha [BH][N], a gate per token
    const uint8_t *slots;  // mode 2: [BH][nchunks] gate slots (GateSlot, 2 KB each)
    float *gprod;          // mode 2: [items] each segment's product of gates
    int *ctrl;          // [0] ticket counter, [1] abort flag
    int *status;        // device status word
    uint16_t *out;      // [BH][N][DK] bf16 output
    long long timeout;  // clock cycles per bounded wait
};

template <int DK, int kMode>
struct Layout {
    static constexpr int KB = DK / 64;
    static constexpr int STAGES = DK == 128 ? 2 : (kMode == 2 ? 3 : 4);
    static constexpr int TILE = DK * C * 2;   // a Q or K tile (bf16)
    static constexpr int VTILE = C * DV * 2;  // a V (or O) tile half
    // mode 2: the chunk's gate prefix and column factors (GateSlot, 1.5 KB,
    // padded to keep every stage 1024-byte aligned) after V
    static constexpr int GS = kMode == 2 ? 2048 : 0;
    static constexpr int OFF_GS = 2 * TILE + VTILE;
    static constexpr int STAGE = 2 * TILE + VTILE + GS;
    static_assert(STAGE % 1024 == 0, "SW128 tiles need 1024-byte aligned stages");
    static constexpr int OFF_Q = 0, OFF_K = TILE, OFF_V = 2 * TILE;
    // [S | z] in bf16: MN-major B operand [K = a][N = 80]; block 0 = S,
    // block 1 column 0 = z (rest zero)
    static constexpr int OFF_SB = STAGES * STAGE;
    static constexpr int SBLK = DK * 128;
    static constexpr int SB = 2 * SBLK;
    // [V | 1]: 64-column block whose column 0 is one (rest zero), the
    // second N block of the V operand (reached through the descriptor LBO)
    static constexpr int OFF_ONESX = OFF_SB + SB;
    static constexpr int ONESX = 16384;
    static constexpr int OFF_SMALL = OFF_ONESX + ONESX;
    static constexpr int STATE = DK * DV + DK;
};

struct Small {
    float gtab[32];  // score epilogue: g^0 .. g^31 of the current head
    uint64_t full[4], empty[4], xf[4];
    uint64_t pfull[2], pt_ready[2], pv_done[2], o_full[2], o_empty[2];
    uint64_t s_full, sb_ready;
    // with weights: chunk nb's Q and K rows carry their weights (two, by the
    // parity of nb: the transform may complete chunk nb + 1 before the MMA
    // issuer has observed chunk nb, never nb + 2, since P(nb + 2) is only
    // issued after that observation)
    uint64_t khat_ready[2];
    uint64_t item_full[2], item_empty[2];
    uint64_t fin;  // every product of the CTA has completed (exit)
    int ring[2];
    int lb_n;  // look-back decision of the current item
    float tg_l[8], eg_l[4];  // mode 2: per-warp gate sums (transform, state roles)
    int tg_z[8], eg_z[4];
    uint32_t tmem_base;
};

// A work item: segment `seg` of head `bh` (value-column half `half`),
// chunks [c0, c1).  Segment 0 spans seg0 chunks, later ones seg_chunks.
// Phase A of segment s >= 1 reduces its predecessor's chunks [a0, a1 = c0)
// to that segment's local state, weighted relative to c0: the first term of
// its own start state, kept in TMEM.  It publishes that state (pub) when a
// later segment needs it too.  Segment 0 starts from zero and runs phase B
// at once.
struct Item {
    int bh, seg, half, c0, c1, a0, a1;
    bool hasA, pub;
};

__device__ __forceinline__ Item decode_item(int t, const Params &p) {
    Item it;
    it.half = t % p.nhalf;
    const int u = t / p.nhalf;
    it.bh = u % p.BH;
    it.seg = u / p.BH;
    it.c0 = it.seg == 0 ? 0 : p.seg0 + (it.seg - 1) * p.seg_chunks;
    it.c1 = min(it.seg == 0 ? p.seg0 : it.c0 + p.seg_chunks, p.nchunks);
    it.a0 = it.seg <= 1 ? 0 : p.seg0 + (it.seg - 2) * p.seg_chunks;
    it.a1 = it.c0;
    it.hasA = it.seg > 0;
    it.pub = it.seg > 0 && it.seg < p.nseg - 1;
    return it;
}

__device__ __forceinline__ int item_index(int bh, int seg, int half,
                                          const Params &p) {
    return (seg * p.BH + bh) * p.nhalf + half;
}

// Pop the next item id from the CTA's item ring (every thread of a role
// calls; `nthreads` threads share the named barrier `bar_id`, or 0 for a
// single-thread role).
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

// ---------------------------------------------------------------- producer

template <int DK, int kMode>
__device__ void producer(uint8_t *smem, Small &sm, const Params &p,
                         const Ctx &cx, const CUtensorMap *tq,
                         const CUtensorMap *tk, const CUtensorMap *tv) {
    using L = Layout<DK, kMode>;
    const uint64_t keep = policy_evict_last(), stream = policy_evict_first();
    int j = 0, tl = 0;
    bool stop = false;  // a wait gave up: no further loads
    for (;;) {
        int t = atomicAdd(p.ctrl, 1);
        if (t >= p.items || stop || *cx.abort) t = -1;
        const int r = tl & 1;
        settle_wait(&sm.item_empty[r], ((tl >> 1) & 1) ^ 1);
        ((volatile int *)sm.ring)[r] = t;
        mbar_arrive(&sm.item_full[r]);
        ++tl;
        if (t < 0) break;
        const Item it = decode_item(t, p);
        (void)LA_DCHECK(p.status, it.bh >= 0 && it.bh < p.BH && it.seg < p.nseg && it.a0 >= 0 &&
                                      it.a0 <= it.a1 && it.a1 == it.c0 && it.c0 < it.c1 &&
                                      it.c1 <= p.nchunks && it.half < p.nhalf);
        for (int pass = it.hasA ? 0 : 1; pass < 2 && !stop; ++pass) {
            const int cb = pass == 0 ? it.a0 : it.c0, ce = pass == 0 ? it.a1 : it.c1;
            for (int c = cb; c < ce; ++c, ++j) {
                const int st = j % L::STAGES;
                const uint32_t par = ((j / L::STAGES) & 1) ^ 1;
                if (!wait_bar(&sm.empty[st], par, cx)) {
                    stop = true;
                    break;
                }
                // one arming per phase: the slot's previous load has landed
                // (it always has unless a wait gave up and let a consumer
                // run ahead)
                if (j >= L::STAGES) settle_wait(&sm.full[st], par);
                uint8_t *base = smem + st * L::STAGE;
                const uint64_t pol = pass == 0 ? keep : stream;
                mbar_arrive_expect_tx(&sm.full[st], (pass == 0 ? L::TILE + L::VTILE
                                                               : 2 * L::TILE + L::VTILE) +
                                                        (kMode == 2 ? kGateSlotBytes : 0));
                if (kMode == 2 &&  // the chunk's gate slot, computed ahead
                    LA_DCHECK(p.status, c >= 0 && c < p.nchunks))
                    bulk_load(base + L::OFF_GS,
                              p.slots + ((size_t)it.bh * p.nchunks + c) * kGateSlotBytes,
                              kGateSlotBytes, &sm.full[st]);
                if (pass == 1)
                    for (int kb = 0; kb < L::KB; ++kb)
                        tma_load_3d(base + L::OFF_Q + kb * 16384, tq, &sm.full[st],
                                    64 * kb, c * C, it.bh, stream);
                for (int kb = 0; kb < L::KB; ++kb)
                    tma_load_3d(base + L::OFF_K + kb * 16384, tk, &sm.full[st],
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

// Mode 2, a data-dependent gate alpha_t per token ("Linear Attention", GLA:
// S_t = G_t (.) S_{t-1} + k_t v_t^T, here with the scalar G_t = alpha_t).
// For the tokens of one chunk, lg2[t] is the sum of log2(alpha_u) over the
// nonzero gates u <= t and nz[t] the number of zero gates u <= t (chunk-local
// inclusive prefixes), so that the product of the gates u = j+1..i is
// (nz[i] == nz[j]) ? 2^(lg2[i] - lg2[j]) : 0 -- exact where a gate is 0.
// Tokens past N count as gate 1.  colf[j] is the product of the gates
// u = j+1 .. e(j), e(j) the last token of j's 32-token block, so that where
// j's block lies wholly before row i's block the product u = j+1..i factors
// into a per-row term (u = e(j)+1..i) times colf[j]; both factors lie in
// [0, 1] and neither overflows.  colg[j] = 2^(lg2[s] - lg2[j]), s the token
// before j's block, serves the diagonal block (row and column in one block)
// where that block has no zero gate and a log2 span within kGateSpan: the
// product is then 2^(lg2[i] - lg2[s]) colg[j], both factors normal floats.
// Every chunk's slot is computed ahead of the forward (gate_slots_kernel);
// the producer copies it into the chunk's stage with its tiles.
struct GateSlot {
    float lg2[C];
    int nz[C];
    float colf[C];
    float colg[C];
};
constexpr float kGateSpan = 100.f;
// Folded weights: a chunk whose weights all lie in range takes Qhat and
// Khat as soon as they are mapped, P from them, and one factor per chunk in
// the score epilogue (see chunk_folds).  Decay: g >= 0.77 (log2 below), so
// that g^(2C-1) >= 2^-96; gates: no zero gate in the chunk and a product of
// at least 2^-48, so that every power in P stays above 2^-96.  Only with
// the elu + 1 feature map: its features are positive, so the bf16 rounding
// of the weighted rows costs P a relative 2^-8 at most; with the identity
// map the terms of q . k cancel and that rounding error would not shrink
// with P.
constexpr float kFoldLog2 = -0.3770f;  // log2(0.77)
constexpr float kFoldGateLog2 = -48.f;
static_assert(sizeof(GateSlot) == kGateSlotBytes, "a gate slot is copied whole");

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Whether chunk weights fold into Q and K (mode 1: per head; mode 2: per
// chunk, from its gate slot), and the factor of P then: Qhat_i . Khat_j =
// w(i) w'(j) phi(q_i) . phi(k_j) = G prod_{u=j+1..i}, with G = g^n or the
// chunk's gate product, so Pt = P / G.
template <int kMode>
__device__ __forceinline__ bool chunk_folds(float lg, const GateSlot &g, int n, int phi) {
    if (!phi) return false;
    if (kMode == 1) return lg >= kFoldLog2;
    if (kMode == 2) return g.nz[n - 1] == 0 && g.lg2[n - 1] >= kFoldGateLog2;
    return false;
}

// ---------------------------------------------------------------- MMA issuer

// P = phi(Q) phi(K)^T of job `jj` (stage jj % STAGES) into P buffer b of
// B-chunk number `nbq`, once the chunk is transformed and the buffer's
// previous P~V has completed.
template <int DK, int kMode>
__device__ __forceinline__ void issue_p(uint8_t *smem, Small &sm, const Ctx &cx,
                                        uint32_t tmem, int jj, int nbq) {
    using L = Layout<DK, kMode>;
    constexpr uint32_t idP = idesc_bf16(128, 128, 0, 0);
    const int st = jj % L::STAGES, b = nbq & 1;
    wait_bar(&sm.xf[st], (jj / L::STAGES) & 1, cx);
    wait_bar(&sm.pv_done[b], ((nbq >> 1) & 1) ^ 1, cx);
    tc_fence_after();
    const uint32_t qb = smem_u32(smem + st * L::STAGE + L::OFF_Q);
    const uint32_t kb = smem_u32(smem + st * L::STAGE + L::OFF_K);
    for (int ks = 0; ks < DK / 16; ++ks) {
        const uint32_t off = kmajor_off(ks, 16384);
        mma_ss(tmem + TM_P + 128u * b, sdesc_sw128(qb + off, 16, 1024),
               sdesc_sw128(kb + off, 16, 1024), idP, ks > 0 ? 1u : 0u);
    }
    mma_commit(&sm.pfull[b]);
}

// Issues P of B chunk qi+1 now if its feature maps and P buffer are ready;
// otherwise it is issued (blocking) at the top of the next chunk, so the
// state-dependent products of chunk qi never wait on the transform.
template <int DK, int kMode>
__device__ __forceinline__ void try_issue_next_p(uint8_t *smem, Small &sm,
                                                 const Ctx &cx, uint32_t tmem,
                                                 int jj, int nbq, int qi,
                                                 int nB, int &p_next) {
    using L = Layout<DK, kMode>;
    if (p_next != qi + 1 || qi + 1 >= nB) return;
    const int st1 = (jj + 1) % L::STAGES, b1 = (nbq + 1) & 1;
    // test_wait never suspends the thread (try_wait may, for a
    // system-dependent time, when the phase is not complete)
    if (mbar_test_wait(&sm.xf[st1], ((jj + 1) / L::STAGES) & 1) &&
        mbar_test_wait(&sm.pv_done[b1], (((nbq + 1) >> 1) & 1) ^ 1)) {
        issue_p<DK, kMode>(smem, sm, cx, tmem, jj + 1, nbq + 1);
        ++p_next;
    }
}

template <int DK, int kMode>
__device__ void mma_issuer(uint8_t *smem, Small &sm, const Params &p,
                           const Ctx &cx, const DecayArgs &dk, uint32_t tmem) {
    using L = Layout<DK, kMode>;
    constexpr uint32_t idPV = idesc_bf16(128, NX, 0, 1);  // Pt [V | 1]
    constexpr uint32_t idQS = idesc_bf16(128, NX, 0, 1);  // phi(Q) [S | z]
    constexpr uint32_t idSU = idesc_bf16(128, NX, 1, 1);  // phi(K)^T [V | 1]
    constexpr uint32_t lboA = DK == 128 ? 16384 : 0;      // d=64: rows 64..127 alias
    // chunk order: phi(Q) [S | z] and the state update first, then P(j+1),
    // then P~V(j): the state half heads the chunk's dependency chain (B4 H16
    // N4096 d64, same process: 48.6 against 50.7 us with P~V first; gated
    // 58.8-60.9 against 60.9-62.9 us)
    const uint32_t sb = smem_u32(smem + L::OFF_SB);
    const uint32_t onesx = smem_u32(smem + L::OFF_ONESX);
    int j = 0, nb = 0, nsb = 0, nk = 0, tl = 0;  // nk: chunks weighted after P
    for (;;) {
        const int t = pop_item(sm, tl, cx, 0, 0, true);
        if (t < 0) break;
        const Item it = decode_item(t, p);
        const float lg = head_log2g(dk, it.bh);
        if (it.hasA) {
            // phase A: the segment's local state.  S's columns are free: the
            // previous item read them before its last sb_ready.  Phase-A
            // stages have no output, so both of their releases come from here.
            for (int c = it.a0; c < it.a1; ++c, ++j) {
                const int st = j % L::STAGES;
                wait_bar(&sm.xf[st], (j / L::STAGES) & 1, cx);
                tc_fence_after();
                const uint32_t kb = smem_u32(smem + st * L::STAGE + L::OFF_K);
                const uint32_t vb = smem_u32(smem + st * L::STAGE + L::OFF_V);
                // Khat^T [V | 1]
                for (int ks = 0; ks < C / 16; ++ks)
                    mma_ss(tmem + TM_S, sdesc_sw128(kb + ks * 2048, lboA, 1024),
                           sdesc_sw128(vb + ks * 2048, onesx - vb, 1024), idSU,
                           (c > it.a0 || ks > 0) ? 1u : 0u);
                if (c == it.a1 - 1) mma_commit(&sm.s_full);
                mma_commit(&sm.empty[st]);
                mma_commit(&sm.empty[st]);
            }
        }
        // phase B.  The state after the item's last chunk is only read when
        // it is the sequence's final state and the caller asked for it;
        // otherwise that chunk has no state update.
        const int nB = it.c1 - it.c0;
        const bool final_state = p.S_out && it.seg == p.nseg - 1;
        int p_next = 0;  // first B chunk of the item whose P is not issued
        for (int qi = 0; qi < nB; ++qi) {
            const int jj = j + qi, nbq = nb + qi;
            const int st = jj % L::STAGES, b = nbq & 1;
            const bool su = qi + 1 < nB || final_state;
            if (p_next == qi) {
                issue_p<DK, kMode>(smem, sm, cx, tmem, jj, nbq);
                ++p_next;
            }
            // whether the chunk's weights fold, read now (its gate slot has
            // landed: P of the chunk is issued) and used after the waits
            // below, so that the load's latency stays off the issue path
            const bool wait_khat =
                kMode && !chunk_folds<kMode>(lg, *reinterpret_cast<const GateSlot *>(
                                                     smem + st * L::STAGE + L::OFF_GS),
                                             min(C, p.N - (it.c0 + qi) * C), p.phi);
            const uint32_t qb = smem_u32(smem + st * L::STAGE + L::OFF_Q);
            const uint32_t kb = smem_u32(smem + st * L::STAGE + L::OFF_K);
            const uint32_t vb = smem_u32(smem + st * L::STAGE + L::OFF_V);
            const int ob = nbq & 1;
            const uint32_t tob = TM_O + 80u * ob;
            wait_bar(&sm.o_empty[ob], ((nbq >> 1) & 1) ^ 1, cx);
            // The state-dependent half first: phi(Q) [S | z] and the
            // state update run while the score epilogue works on P(j).
            wait_bar(&sm.sb_ready, nsb & 1, cx);
            ++nsb;
            // with weights: Qhat_i = g^(i+1) phi(q_i) and Khat_t =
            // g^(n-1-t) phi(k_t) (or the products of gates) in place,
            // once P(j) has read the unweighted rows
            if (wait_khat) {
                wait_bar(&sm.khat_ready[nk & 1], (nk >> 1) & 1, cx);
                ++nk;
            }
            tc_fence_after();
            // inter-chunk read phi(Q) [S | z] (Qhat with weights)
            for (int ks = 0; ks < DK / 16; ++ks)
                mma_ss(tmem + tob, sdesc_sw128(qb + kmajor_off(ks, 16384), 16, 1024),
                       sdesc_sw128(sb + ks * 2048, L::SBLK, 1024), idQS,
                       ks > 0 ? 1u : 0u);
            // state update phi(K)^T [V | 1] (Khat with weights)
            if (su) {
                for (int ks = 0; ks < C / 16; ++ks)
                    mma_ss(tmem + TM_S, sdesc_sw128(kb + ks * 2048, lboA, 1024),
                           sdesc_sw128(vb + ks * 2048, onesx - vb, 1024), idSU, 1u);
                mma_commit(&sm.s_full);
            }
            try_issue_next_p<DK, kMode>(smem, sm, cx, tmem, jj, nbq, qi, nB, p_next);
            wait_bar(&sm.pt_ready[b], (nbq >> 1) & 1, cx);
            tc_fence_after();
            // intra-chunk: P~ [V | 1] (P~ read from TMEM)
            for (int ks = 0; ks < C / 16; ++ks)
                mma_ts(tmem + tob, tmem + TM_P + 128u * b + ks * 8,
                       sdesc_sw128(vb + ks * 2048, onesx - vb, 1024), idPV, 1u);
            mma_commit(&sm.o_full[ob]);
            mma_commit(&sm.pv_done[b]);
            // the stage: one release per consumer (the output epilogue
            // gives the second)
            mma_commit(&sm.empty[st]);
        }
        if (final_state) {
            // S's columns are reused by the next item: wait until the
            // output warpgroup has read the final state
            wait_bar(&sm.sb_ready, nsb & 1, cx);
            ++nsb;
        }
        j += nB;
        nb += nB;
    }
    // every product has completed before TMEM is released
    mma_commit(&sm.fin);
    settle_wait(&sm.fin, 0);
}

// ---------------------------------------------------------------- gates (mode 2)

// prod_{u=j+1..i} alpha_u within a chunk (j < i; j = -1: from the chunk's
// first token, i.e. prod_{u<=i}).
__device__ __forceinline__ float gate_prod(const GateSlot &g, int i, int j) {
    const float lj = j < 0 ? 0.f : g.lg2[j];
    const int zj = j < 0 ? 0 : g.nz[j];
    return g.nz[i] == zj ? fast_exp2(g.lg2[i] - lj) : 0.f;
}

// log2 and zero count of one gate value
__device__ __forceinline__ void gate_terms(float a, float &l, int &z) {
    if (a > 0.f) {
        l = __log2f(a);
        z = 0;
    } else {
        l = 0.f;
        z = 1;
    }
}

// The gate slot of chunk c of head bh (block bh * nchunks + c), one thread
// per token (tokens past N count as gate 1), for every chunk at once ahead
// of the forward kernel: the chunk-local inclusive prefixes of the log2 of
// the nonzero gates and of the zero-gate count, then the column factors
// (see GateSlot).  The blocks also clear the forward's ticket counter and
// flags (nclr 16-byte words at clr), and let the forward kernel start its
// prologue early: it waits for this kernel's completion before it reads
// anything.
__global__ void __launch_bounds__(C) gate_slots_kernel(const float *gates, int N, int nchunks,
                                                       GateSlot *slots, uint4 *clr, size_t nclr) {
    grid_dep_launch();
    __shared__ float wl[C / 32], s_l[C];
    __shared__ int wz[C / 32], s_z[C];
    const int c = (int)(blockIdx.x % (unsigned)nchunks), bh = (int)(blockIdx.x / (unsigned)nchunks);
    const int et = threadIdx.x, lane = et & 31, w = et >> 5;
    for (size_t i = (size_t)blockIdx.x * C + et; i < nclr; i += (size_t)gridDim.x * C)
        clr[i] = make_uint4(0u, 0u, 0u, 0u);
    const int tok = c * C + et;
    const float a = tok < N ? __ldg(gates + (size_t)bh * N + tok) : 1.f;
    float l;
    int z;
    gate_terms(a, l, z);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float lo = __shfl_up_sync(~0u, l, o);
        const int zo = __shfl_up_sync(~0u, z, o);
        if (lane >= o) {
            l += lo;
            z += zo;
        }
    }
    if (lane == 31) {
        wl[w] = l;
        wz[w] = z;
    }
    __syncthreads();
    for (int w2 = 0; w2 < w; ++w2) {
        l += wl[w2];
        z += wz[w2];
    }
    s_l[et] = l;
    s_z[et] = z;
    __syncthreads();
    GateSlot &g = slots[(size_t)bh * nchunks + c];
    const int e = et | 31, s = (et & ~31) - 1;
    g.lg2[et] = l;
    g.nz[et] = z;
    g.colf[et] = s_z[e] == z ? fast_exp2(s_l[e] - l) : 0.f;
    // >= 1; clamped, as blocks past the span never read it
    g.colg[et] = fast_exp2(fminf((s < 0 ? 0.f : s_l[s]) - l, kGateSpan + 1.f));
}

// Totals over tokens [t0, t1) of head bh: sum of log2 of the nonzero gates
// and the number of zero gates (`nthr` threads of one role, `tid` 0-based,
// scratch `sl`/`sz` with one entry per warp, named barrier `bar`).
__device__ __forceinline__ void gate_totals(float &L2, int &Z, const Params &p,
                                            int bh, int t0, int t1, int tid,
                                            int nthr, float *sl, int *sz, int bar) {
    float l = 0.f;
    int z = 0;
    const float *ga = p.gates + (size_t)bh * p.N;
    // eight loads in flight per thread before any is used
    constexpr int kBatch = 8;
    for (int t = t0 + tid; t < t1; t += kBatch * nthr) {
        float a[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int tok = t + u * nthr;
            a[u] = tok < t1 ? __ldg(ga + tok) : 1.f;
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            float lt;
            int zt;
            gate_terms(a[u], lt, zt);
            l += lt;
            z += zt;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        l += __shfl_xor_sync(~0u, l, o);
        z += __shfl_xor_sync(~0u, z, o);
    }
    if ((tid & 31) == 0) {
        sl[tid >> 5] = l;
        sz[tid >> 5] = z;
    }
    named_bar_sync(bar, nthr);
    L2 = 0.f;
    Z = 0;
    for (int w = 0; w < nthr / 32; ++w) {
        L2 += sl[w];
        Z += sz[w];
    }
    named_bar_sync(bar, nthr);
}

// ---------------------------------------------------------------- transform

// In place in stage `st`, once P of that chunk (`nb`, the only reader of the
// unweighted rows) has completed: Khat_t = g^(n-1-t) phi(k_t), the weight of
// token t in the state after the chunk (rows past N are zero), and
// Qhat_i = g^(i+1) phi(q_i), the weight of the chunk's start state in row i;
// with gates prod_{u=t+1..n-1} alpha_u and prod_{u<=i} alpha_u.  The
// inter-chunk read Qhat [S | z] then accumulates onto P~ [V | 1] directly.
// All transform threads call, for the chunks that do not fold only (a
// folded chunk was weighted when it was mapped, and the MMA issuer does not
// wait for it).  khat_ready is indexed by the count `nk` of such chunks; the
// wait on P(nb) keeps the transform from arriving twice on one barrier
// before the MMA issuer has observed the first arrival.
template <int DK, int kMode>
__device__ __forceinline__ void weight_qk(uint8_t *smem, Small &sm, const Ctx &cx,
                                          float lg, int st, int n, int nb, int nk,
                                          int row, int part, int et) {
    using L = Layout<DK, kMode>;
    wait_bar(&sm.pfull[nb & 1], (nb >> 1) & 1, cx);
    const GateSlot &g = *reinterpret_cast<const GateSlot *>(smem + st * L::STAGE + L::OFF_GS);
    const float wk = row >= n ? 0.f
                              : (kMode == 2 ? gate_prod(g, n - 1, row) : gpow(lg, n - 1 - row));
    const float wq = kMode == 2 ? gate_prod(g, row, -1) : gpow(lg, row + 1);
    scale_row<DK>(smem + st * L::STAGE + L::OFF_K, row, part, bf2_splat(wk));
    scale_row<DK>(smem + st * L::STAGE + L::OFF_Q, row, part, bf2_splat(wq));
    fence_async_shared();
    named_bar_sync(BAR_T, kTThreads);
    if (et == 0) mbar_arrive(&sm.khat_ready[nk & 1]);
}

template <int DK, int kMode>
__device__ void transform(uint8_t *smem, Small &sm, const Params &p,
                          const Ctx &cx, const DecayArgs &dk) {
    using L = Layout<DK, kMode>;
    const int et = threadIdx.x - kWarpT * 32;  // 0..255
    const int row = et & 127, part = et >> 7;
    int j = 0, nb = 0, nk = 0, tl = 0;  // nk: chunks weighted after P (not folded)
    for (;;) {
        const int t = pop_item(sm, tl, cx, BAR_T, kTThreads, et == 0);
        if (t < 0) break;
        const Item it = decode_item(t, p);
        const float lg = head_log2g(dk, it.bh);
        if (it.hasA) {
            // phase A over the predecessor's chunks [a0, a1): Khat_t =
            // g^(a1 C - 1 - t) phi(k_t), t relative to the end of that range
            // (the item's own start); with gates Khat_t = prod_{u>t in the
            // range} alpha_u phi(k_t).  Every chunk of the range is full.
            const int seg_end = it.a1 * C;
            float L2 = 0.f, off2 = 0.f;
            int Z = 0, offz = 0;
            if (kMode == 2)
                gate_totals(L2, Z, p, it.bh, it.a0 * C, seg_end, et, kTThreads,
                            sm.tg_l, sm.tg_z, BAR_T);
            for (int c = it.a0; c < it.a1; ++c, ++j) {
                const int st = j % L::STAGES;
                wait_bar(&sm.full[st], (j / L::STAGES) & 1, cx);
                uint8_t *kt = smem + st * L::STAGE + L::OFF_K;
                const int tok = c * C + row;
                if (kMode || tok >= p.N) {
                    float w;
                    if (kMode == 2) {
                        const GateSlot &g =
                            *reinterpret_cast<const GateSlot *>(smem + st * L::STAGE + L::OFF_GS);
                        w = tok < p.N && Z == offz + g.nz[row]
                                ? fast_exp2(L2 - (off2 + g.lg2[row])) : 0.f;
                        const int nv = min(C, p.N - c * C);
                        off2 += g.lg2[nv - 1];
                        offz += g.nz[nv - 1];
                    } else {
                        w = tok < p.N ? gpow(lg, seg_end - 1 - tok) : 0.f;
                    }
                    transform_row_scaled<DK>(kt, row, part, bf2_splat(w), p.phi);
                } else {
                    transform_row<DK>(kt, row, part, false, p.phi);
                }
                fence_async_shared();
                named_bar_sync(BAR_T, kTThreads);
                if (et == 0) mbar_arrive(&sm.xf[st]);
            }
        }
        // With weights, chunk c's Q and K rows are weighted in place once
        // P(c) has read them.  With three or more stages that step runs
        // after the feature map of chunk c + 1, so the feature map overlaps
        // P(c); with two, chunk c + 1's stage is chunk c - 1's, whose
        // release would then sit on the path, so it runs at once.
        constexpr bool kPipe = L::STAGES >= 3;
        int pst = -1, pn = 0, pnb = 0, pnk = 0;
        for (int c = it.c0; c < it.c1; ++c, ++j, ++nb) {
            const int st = j % L::STAGES;
            wait_bar(&sm.full[st], (j / L::STAGES) & 1, cx);
            uint8_t *qt = smem + st * L::STAGE + L::OFF_Q;
            uint8_t *kt = smem + st * L::STAGE + L::OFF_K;
            const int n = min(C, p.N - c * C);
            const GateSlot &g =
                *reinterpret_cast<const GateSlot *>(smem + st * L::STAGE + L::OFF_GS);
            const bool fold = chunk_folds<kMode>(lg, g, n, p.phi);
            if (fold) {
                // Qhat and Khat at once (rows past N -> 0)
                const float wk = row >= n ? 0.f
                                          : (kMode == 2 ? gate_prod(g, n - 1, row)
                                                        : gpow(lg, n - 1 - row));
                const float wq = kMode == 2 ? gate_prod(g, row, -1) : gpow(lg, row + 1);
                transform_row_scaled<DK>(qt, row, part, bf2_splat(wq), p.phi);
                transform_row_scaled<DK>(kt, row, part, bf2_splat(wk), p.phi);
            } else {
                transform_row<DK>(qt, row, part, false, p.phi);
                transform_row<DK>(kt, row, part, row >= n, p.phi);  // rows past N -> 0
            }
            fence_async_shared();
            named_bar_sync(BAR_T, kTThreads);
            if (et == 0) mbar_arrive(&sm.xf[st]);
            if (kMode && !kPipe && !fold)
                weight_qk<DK, kMode>(smem, sm, cx, lg, st, n, nb, nk++, row, part, et);
            if (kMode && kPipe) {
                if (pst >= 0)
                    weight_qk<DK, kMode>(smem, sm, cx, lg, pst, pn, pnb, pnk, row, part, et);
                pst = -1;
                if (!fold) {
                    pst = st;
                    pn = n;
                    pnb = nb;
                    pnk = nk++;
                }
            }
        }
        if (kMode && pst >= 0)
            weight_qk<DK, kMode>(smem, sm, cx, lg, pst, pn, pnb, pnk, row, part, et);
    }
}

// ---------------------------------------------------------------- score epilogue

// Causal mask and decay on P (fp32, TMEM), rounded to bf16 in place (the A
// operand of P~V).  One thread per row i (= TMEM lane).
template <int DK, int kMode>
__device__ void score_epilogue(uint8_t *smem, Small &sm, const Params &p,
                               const Ctx &cx, const DecayArgs &dk, uint32_t tmem) {
    using L = Layout<DK, kMode>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int et = threadIdx.x - kWarpE1 * 32;
    const uint32_t lb = tmem + ((uint32_t)(q * 32) << 16);
    int nb = 0, tl = 0, j = 0;
    for (;;) {
        const int t = pop_item(sm, tl, cx, BAR_E1, 128, et == 0);
        if (t < 0) break;
        const Item it = decode_item(t, p);
        const float lg = head_log2g(dk, it.bh);
        if (kMode == 1) {
            if (et < 32) sm.gtab[et] = gpow(lg, et);
            named_bar_sync(BAR_E1, 128);
        }
        if (it.hasA) j += it.a1 - it.a0;  // phase-A jobs
        for (int c = it.c0; c < it.c1; ++c, ++nb, ++j) {
            const int b = nb & 1;
            const uint32_t tp = lb + TM_P + 128u * b;
            wait_bar(&sm.pfull[b], (nb >> 1) & 1, cx);
            tc_fence_after();
            const GateSlot &gs = *reinterpret_cast<const GateSlot *>(
                smem + (j % L::STAGES) * L::STAGE + L::OFF_GS);
            float gl_i = 0.f;
            int gz_i = 0;
            if (kMode == 2) {
                // the chunk's gate prefix (written before the stage's xf)
                wait_bar(&sm.xf[j % L::STAGES], (j / L::STAGES) & 1, cx);
                gl_i = gs.lg2[row];
                gz_i = gs.nz[row];
            }
            // folded weights: P holds G x the weighted scores (G = g^n or
            // the chunk's gate product), so every entry takes 1 / G
            const int n = min(C, p.N - c * C);
            const bool fold = chunk_folds<kMode>(lg, gs, n, p.phi);
            float F = 1.f;
            if (fold) F = kMode == 2 ? fast_exp2(-gs.lg2[n - 1]) : exp2f(-lg * (float)n);
            // not unrolled: the gated paths make four copies of this body
            // too much code for the instruction cache the roles share
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
                    if (fold) {
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            const bool in0 = blk < q || e <= lane, in1 = blk < q || e + 1 <= lane;
                            pk[e >> 1] = pack_bf16x2(in0 ? u2f(v[e]) * F : 0.f,
                                                     in1 ? u2f(v[e + 1]) * F : 0.f);
                        }
                    } else if (blk < q) {
                        if (kMode == 2) {
                            // prod_{u=col+1..row} alpha_u = (prod over
                            // u = e+1..row) colf[col], e the block's last token
                            const int e = 32 * blk + 31;
                            const float base = gz_i == gs.nz[e] ? fast_exp2(gl_i - gs.lg2[e]) : 0.f;
#pragma unroll
                            for (int e2 = 0; e2 < 32; e2 += 2)
                                pk[e2 >> 1] = pack_bf16x2(
                                    u2f(v[e2]) * (base * gs.colf[32 * blk + e2]),
                                    u2f(v[e2 + 1]) * (base * gs.colf[32 * blk + e2 + 1]));
                        } else if (kMode) {
                            // g^(row - j) = g^(row - 32 blk - 31) g^(31 - e)
                            const float base = gpow(lg, row - 32 * blk - 31);
#pragma unroll
                            for (int e = 0; e < 32; e += 2)
                                pk[e >> 1] = pack_bf16x2(
                                    u2f(v[e]) * (base * sm.gtab[31 - e]),
                                    u2f(v[e + 1]) * (base * sm.gtab[30 - e]));
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; e += 2)
                                pk[e >> 1] = pack_bf16x2(u2f(v[e]), u2f(v[e + 1]));
                        }
                    } else if (kMode == 2) {
                        // diagonal block: prod_{u=col+1..row} alpha_u, only
                        // where col <= row.  s is the token before the block.
                        const int s = 32 * blk - 1, eb = 32 * blk + 31;
                        const float ls = s < 0 ? 0.f : gs.lg2[s];
                        const int zs = s < 0 ? 0 : gs.nz[s];
                        if (gs.nz[eb] == zs && ls - gs.lg2[eb] <= kGateSpan) {
                            // no zero gate, span in range (warp-uniform)
                            const float rf = fast_exp2(gl_i - ls);
#pragma unroll
                            for (int e = 0; e < 32; e += 2) {
                                const float x0 = e <= lane
                                    ? u2f(v[e]) * (rf * gs.colg[32 * blk + e]) : 0.f;
                                const float x1 = e + 1 <= lane
                                    ? u2f(v[e + 1]) * (rf * gs.colg[32 * blk + e + 1]) : 0.f;
                                pk[e >> 1] = pack_bf16x2(x0, x1);
                            }
                        } else {
#pragma unroll
                            for (int e = 0; e < 32; e += 2) {
                                const int c0 = 32 * blk + e;
                                const float a0 = fast_exp2(fminf(gl_i - gs.lg2[c0], 0.f));
                                const float a1 = fast_exp2(fminf(gl_i - gs.lg2[c0 + 1], 0.f));
                                const float x0 = e <= lane && gz_i == gs.nz[c0]
                                    ? u2f(v[e]) * a0 : 0.f;
                                const float x1 = e + 1 <= lane && gz_i == gs.nz[c0 + 1]
                                    ? u2f(v[e + 1]) * a1 : 0.f;
                                pk[e >> 1] = pack_bf16x2(x0, x1);
                            }
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; e += 2) {
                            // diagonal block: g^(i - j) = g^(lane - e), from
                            // the head's table, only where e <= lane
                            float x0 = 0.f, x1 = 0.f;
                            if (e <= lane)
                                x0 = kMode ? u2f(v[e]) * sm.gtab[lane - e] : u2f(v[e]);
                            if (e + 1 <= lane)
                                x1 = kMode ? u2f(v[e + 1]) * sm.gtab[lane - e - 1]
                                            : u2f(v[e + 1]);
                            pk[e >> 1] = pack_bf16x2(x0, x1);
                        }
                    }
                }
                tmem_st16(tp + 16 * blk, pk);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&sm.pt_ready[b]);  // 128 arrivals, one per row
        }
    }
}

// One chunk's output: O / den (O alone without the normaliser) in bf16,
// stored to global memory from registers, one token row per thread in
// 16-byte streaming stores (rows past N dropped).  Nothing is staged in
// shared memory, so the chunk's stage goes back to the producer as soon as
// its products have completed.
template <int DK, int kMode>
__device__ __forceinline__ void output_chunk(Small &sm, const Params &p, const Ctx &cx,
                                             uint32_t lb, int row, int et, const Item &it,
                                             int c, int j, int nb) {
    using L = Layout<DK, kMode>;
    const int st = j % L::STAGES;
    const int ob = nb & 1;
    const uint32_t tob = TM_O + 80u * ob;
    wait_bar(&sm.o_full[ob], (nb >> 1) & 1, cx);
    tc_fence_after();
    // the output needs nothing from the stage: its second release (the MMA
    // issuer's commit is the first, once the chunk's products completed)
    if (et == 0) mbar_arrive(&sm.empty[st]);
    const int tok = c * C + row;
    const bool live = tok < p.N && LA_DCHECK(p.status, it.bh < p.BH && 64 * it.half < DK);
    uint4 *dst = reinterpret_cast<uint4 *>(p.out) +
                 (((size_t)it.bh * p.N + (live ? tok : 0)) * DK + 64 * it.half) / 8;
    uint32_t dreg = tmem_ld1(lb + tob + DV);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t o[32];
        tmem_ld32(lb + tob + 32 * h, o);
        tmem_wait_ld();
        reg_fence(o);
        reg_fence(dreg);
        const float inv = p.norm ? 1.f / u2f(dreg) : 1.f;
        if (h == 1) {
            tc_fence_before();
            mbar_arrive(&sm.o_empty[ob]);  // 128 arrivals: O has been read
        }
        if (live) {
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
                __stcs(dst + 4 * h + ch,
                       make_uint4(pack_bf16x2(u2f(o[8 * ch]) * inv, u2f(o[8 * ch + 1]) * inv),
                                  pack_bf16x2(u2f(o[8 * ch + 2]) * inv, u2f(o[8 * ch + 3]) * inv),
                                  pack_bf16x2(u2f(o[8 * ch + 4]) * inv, u2f(o[8 * ch + 5]) * inv),
                                  pack_bf16x2(u2f(o[8 * ch + 6]) * inv, u2f(o[8 * ch + 7]) * inv)));
        }
    }
}

// ---------------------------------------------------------------- output + state

// Output epilogue (O / den, bf16, stored from registers) and state epilogue (bf16 [S | z]
// operand of the next chunk, decay rescale, segment publication and
// look-back) on one warpgroup.  Per chunk j the state of chunk j+1 is
// prepared first (it gates the next phi(Q) [S | z]), then chunk j's output.

// Writes bf16 values of one 32-column half of S row `a` into block 0 of the
// [S | z] operand (MN-major, K = a rows).
__device__ __forceinline__ void store_sb_half(uint8_t *sb, int a, int h,
                                              const float (&x)[32]) {
#pragma unroll
    for (int ch = 0; ch < 4; ++ch)
        *reinterpret_cast<uint4 *>(sb + sw128_offset(a, 32 * h + ch * 8)) =
            make_uint4(pack_bf16x2(x[8 * ch], x[8 * ch + 1]),
                       pack_bf16x2(x[8 * ch + 2], x[8 * ch + 3]),
                       pack_bf16x2(x[8 * ch + 4], x[8 * ch + 5]),
                       pack_bf16x2(x[8 * ch + 6], x[8 * ch + 7]));
}

// z[a] in bf16 at column 0 of block 1 of the [S | z] operand.
__device__ __forceinline__ void store_zb(uint8_t *sb_z, int a, float z) {
    *reinterpret_cast<__nv_bfloat16 *>(sb_z + sw128_offset(a, 0)) =
        __float2bfloat16_rn(z);
}

// z column of the [S | z] accumulator: (z, 0, ..., 0) over 16 columns.
__device__ __forceinline__ void tmem_put_z(uint32_t taddr, float z) {
    uint32_t v[16];
    v[0] = __float_as_uint(z);
#pragma unroll
    for (int e = 1; e < 16; ++e) v[e] = 0u;
    tmem_st16(taddr, v);
}

// State-epilogue thread mapping.  For d = 64 the state accumulator's lanes
// 64..127 hold a copy of rows 0..63 (the A operand's rows alias), so lanes
// 0..63 take columns 0..31 and lanes 64..127 columns 32..63 of the same
// rows, and every thread of the warpgroup has work; for d = 128 each lane is
// one row and takes both 32-column halves.  z goes with column half 0.
template <int DK>
struct SMap {
    static constexpr int NH = DK == 64 ? 1 : 2;  // halves per thread
    int a, h0;
    bool hasz;
    __device__ __forceinline__ explicit SMap(int lane)
        : a(DK == 64 ? (lane & 63) : lane), h0(DK == 64 ? (lane >> 6) : 0),
          hasz(DK == 64 ? lane < 64 : true) {}
};

// Look-back, step 1 (one warp): decided once segments 1 .. seg-1 of the
// head and half (which hold the local states of segments 0 .. seg-2) have
// all published; 32 flags per look.  Leaves seg - 1 in lb_n, or -1 when
// `wait` is false and one of them has not published yet.
__device__ __forceinline__ void resolve_lookback(Small &sm, const Params &p,
                                                 const Item &it, const Ctx &cx,
                                                 int lane, bool wait) {
    int n = it.seg > 0 ? it.seg - 1 : 0;
    long long dl = 0;
    for (int base = 1; base < it.seg && n >= 0; base += 32) {
        const int s = base + lane;
        const int fi = item_index(it.bh, s < it.seg ? s : 1, it.half, p);
        const bool ok = LA_DCHECK(p.status, fi >= 0 && fi < p.items);
        const int *fp = p.flags + (ok ? fi : 0);
        for (;;) {
            const int f = s < it.seg && ok ? load_flag(fp) : FLAG_AGG;
            if (__all_sync(~0u, f >= FLAG_AGG)) break;
            if (!wait) {
                n = -1;
                break;
            }
            if (__any_sync(~0u, *cx.abort != 0)) {
                base = it.seg;  // aborted: the kernel finishes with invalid output
                break;
            }
            const long long now = __shfl_sync(~0u, clock64(), 0);
            if (dl == 0) {
                dl = now + cx.timeout;
            } else if (now > dl) {
                if (lane == 0)
                    raise_timeout(cx, 0x80000u | ((uint32_t)(reinterpret_cast<uintptr_t>(fp) >> 2) & 0x7FFFFu));
                base = it.seg;
                break;
            }
            __nanosleep(64);
        }
    }
    if (lane == 0) sm.lb_n = n;
}

// Look-back, step 2 (every thread): its 32 columns (half h) of row a of
// sum_{m = 0..nlb-1} w_m local(seg-2-m), nearest first (a fixed order, so
// the start state does not depend on timing), and z[a].  local(j) is in the
// slot of segment j + 1.  w_0 = w0 is the decay across the item's own
// phase-A range (segment seg-1); each further term is decayed across one more
// segment: g^(L C), or with gates the product its holder published.
template <int DK, int kMode>
__device__ __forceinline__ void lookback_sum(const Small &sm, const Params &p,
                                             const Item &it, int nlb, int a,
                                             int h, bool zh, float gL, float w0,
                                             float (&acc)[32], float &accz) {
    using L = Layout<DK, kMode>;
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] = 0.f;
    accz = 0.f;
    float w = w0;
    for (int m = 0; m < nlb; ++m) {
        const int pi = item_index(it.bh, it.seg - 1 - m, it.half, p);
        if (!LA_DCHECK(p.status, pi >= 0 && pi < p.items && a >= 0 && a < DK && h >= 0 &&
                                     32 * h + 32 <= DV))
            continue;
        const float *src = p.agg + (size_t)pi * L::STATE;
        const float4 *s4 = reinterpret_cast<const float4 *>(src + a * DV + 32 * h);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float4 u = __ldcg(s4 + e);
            acc[4 * e] = fmaf(w, u.x, acc[4 * e]);
            acc[4 * e + 1] = fmaf(w, u.y, acc[4 * e + 1]);
            acc[4 * e + 2] = fmaf(w, u.z, acc[4 * e + 2]);
            acc[4 * e + 3] = fmaf(w, u.w, acc[4 * e + 3]);
        }
        if (zh) accz = fmaf(w, __ldcg(src + DK * DV + a), accz);
        w *= kMode == 2 ? __ldcg(p.gprod + pi) : gL;
    }
}

// The item's own phase-A result (TMEM S, this thread's 32 columns of half
// h, and z[a]) added to a look-back sum: the start state's first term.
__device__ __forceinline__ void add_own_state(uint32_t lb, int h, bool zh,
                                              float (&acc)[32], float &accz) {
    uint32_t v[32];
    tmem_ld32(lb + TM_S + 32 * h, v);
    tmem_wait_ld();
    reg_fence(v);
#pragma unroll
    for (int e = 0; e < 32; ++e) acc[e] = u2f(v[e]) + acc[e];
    if (zh) {
        uint32_t zl = tmem_ld1(lb + TM_S + DV);
        tmem_wait_ld();
        reg_fence(zl);
        accz = u2f(zl) + accz;
    }
}

// A thread's fp32 slot for half hh of its look-back sum, parked in the
// [S | z] operand buffer (idle between an item's start and its phase B):
// one 128-byte row of the buffer, the one the thread itself rewrites in
// bf16 afterwards where possible (d = 128: block hh, row a; d = 64: block
// 1 - h0, row a, shared with the row's other thread, so there the rewrite
// waits for a barrier).  16-byte pieces rotate with the row (no bank
// conflicts).
template <int DK>
__device__ __forceinline__ float4 *lb_slot(uint8_t *sb, int a, int h0, int hh) {
    const int blk = DK == 128 ? hh : 1 - h0;
    return reinterpret_cast<float4 *>(sb + blk * (DK * 128) + a * 128);
}

// Row a of block 1 of the [S | z] operand: z[a] in column 0, zero elsewhere.
__device__ __forceinline__ void store_zrow(uint8_t *sb_z, int a, float z) {
    uint4 *row = reinterpret_cast<uint4 *>(sb_z + a * 128);
#pragma unroll
    for (int c = 0; c < 8; ++c) row[c] = make_uint4(0u, 0u, 0u, 0u);
    store_zb(sb_z, a, z);
}

template <int DK, int kMode>
__device__ void output_state(uint8_t *smem, Small &sm, const Params &p,
                             const Ctx &cx, const DecayArgs &dk, uint32_t tmem) {
    using L = Layout<DK, kMode>;
    using SM = SMap<DK>;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;
    const int et = threadIdx.x - kWarpE2 * 32;
    const int ln = q * 32 + lane;  // the TMEM lane this thread may access
    const SM sm_map(ln);
    const int a = sm_map.a, h0 = sm_map.h0;
    const bool hasz = sm_map.hasz;
    const uint32_t lb = tmem + ((uint32_t)(q * 32) << 16);  // lanes of this warp
    uint8_t *sb = smem + L::OFF_SB;
    uint8_t *sbz = sb + L::SBLK;
    const int row = ln;  // output row i
    int tl = 0, ns = 0, j = 0, nb = 0;
    for (;;) {
        const int t = pop_item(sm, tl, cx, BAR_E2, 128, et == 0);
        if (t < 0) break;
        const Item it = decode_item(t, p);
        const float lg = head_log2g(dk, it.bh);
        // The decay across one segment of seg_chunks chunks: every segment a
        // look-back reaches across (1 .. seg-1) has that length.  w0 is the
        // decay across the item's own phase-A range; with gates the product
        // of its gates, published with the state for the segments after it.
        const float gL = gpow(lg, p.seg_chunks * C);
        float w0 = gL;
        if (kMode == 2 && it.hasA) {
            float L2;
            int Z;
            gate_totals(L2, Z, p, it.bh, it.a0 * C, it.a1 * C, et, 128,
                        sm.eg_l, sm.eg_z, BAR_E2);
            w0 = Z == 0 ? exp2f(L2) : 0.f;
            if (et == 0 && it.pub && LA_DCHECK(p.status, t < p.items))
                p.gprod[t] = w0;  // visible with the item's flags
        }
        float *agg = p.agg + (size_t)t * L::STATE;
        const int n0 = min(C, p.N - it.c0 * C);
        float f0 = gpow(lg, n0);
        // The start state: the item's own phase-A result (TMEM S) plus the
        // states that segments 1 .. seg-1 published.  Look-back, first try:
        // if those have already published, sum them now, while phase A
        // runs, into the threads' slots.
        const bool lbk = it.seg >= 2;
        bool early = false;
        float accz_e = 0.f;
        if (lbk) {
            if (warp == kWarpE2) resolve_lookback(sm, p, it, cx, lane, false);
            named_bar_sync(BAR_E2, 128);
            const int nlb = sm.lb_n;
            early = nlb >= 0;
            if (early) {
#pragma unroll 1
                for (int hh = 0; hh < SM::NH; ++hh) {
                    float acc[32], accz;
                    lookback_sum<DK, kMode>(sm, p, it, nlb, a, h0 + hh,
                                             hasz && hh == 0, gL, w0, acc, accz);
                    if (hh == 0) accz_e = accz;
                    float4 *slot = lb_slot<DK>(sb, a, h0, hh);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        slot[e ^ (a & 7)] = make_float4(acc[4 * e], acc[4 * e + 1],
                                                        acc[4 * e + 2], acc[4 * e + 3]);
                }
            }
        }
        if (it.hasA) {
            j += it.a1 - it.a0;  // the phase-A jobs (released by the MMA issuer)
            wait_bar(&sm.s_full, ns & 1, cx);
            ++ns;
            tc_fence_after();
            if (it.pub) {
                // publish the predecessor's local state at once (a debug
                // check guards the stores only: every thread still reaches
                // the barrier)
                const bool okp = LA_DCHECK(p.status, t < p.items && a < DK);
#pragma unroll
                for (int hh = 0; hh < SM::NH; ++hh) {
                    const int h = h0 + hh;
                    uint32_t v[32];
                    tmem_ld32(lb + TM_S + 32 * h, v);
                    tmem_wait_ld();
                    reg_fence(v);
                    float4 *dst = reinterpret_cast<float4 *>(agg + a * DV + 32 * h);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        if (okp)
                            dst[e] = make_float4(u2f(v[4 * e]), u2f(v[4 * e + 1]),
                                                 u2f(v[4 * e + 2]), u2f(v[4 * e + 3]));
                }
                if (hasz) {
                    uint32_t zl = tmem_ld1(lb + TM_S + DV);
                    tmem_wait_ld();
                    reg_fence(zl);
                    if (okp) agg[DK * DV + a] = u2f(zl);
                }
                __threadfence();
                named_bar_sync(BAR_E2, 128);
                if (et == 0 && okp) publish_flag(p.flags + t, FLAG_AGG);
            }
        }
        if (kMode == 2) {
            // the first chunk's product of gates, from its gate slot (copied
            // in with the chunk's tiles)
            wait_bar(&sm.full[j % L::STAGES], (j / L::STAGES) & 1, cx);
            f0 = gate_prod(*reinterpret_cast<const GateSlot *>(
                               smem + (j % L::STAGES) * L::STAGE + L::OFF_GS),
                           n0 - 1, -1);
        }
        if (early) {
            // the phase-B start state from the sums parked during phase A
#pragma unroll 1
            for (int hh = 0; hh < SM::NH; ++hh) {
                const int h = h0 + hh;
                const bool zh = hasz && hh == 0;
                float acc[32];
                const float4 *slot = lb_slot<DK>(sb, a, h0, hh);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 u = slot[e ^ (a & 7)];
                    acc[4 * e] = u.x;
                    acc[4 * e + 1] = u.y;
                    acc[4 * e + 2] = u.z;
                    acc[4 * e + 3] = u.w;
                }
                float accz = zh ? accz_e : 0.f;
                add_own_state(lb, h, zh, acc, accz);
                if (zh) accz_e = accz;
                uint32_t v[32];
                if (zh) tmem_put_z(lb + TM_S + DV, f0 * accz);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(f0 * acc[e]);
                tmem_st32(lb + TM_S + 32 * h, v);
                if (DK == 64) named_bar_sync(BAR_E2, 128);  // every slot read
                store_sb_half(sb, a, h, acc);
                tmem_wait_st();
            }
            if (hasz) store_zrow(sbz, a, accz_e);
        } else {
            // look-back, waiting for segments 1 .. seg-1
            int nlb = 0;
            if (lbk) {
                if (warp == kWarpE2) resolve_lookback(sm, p, it, cx, lane, true);
                named_bar_sync(BAR_E2, 128);
                nlb = sm.lb_n;
            }
#pragma unroll 1
            for (int hh = 0; hh < SM::NH; ++hh) {
                const int h = h0 + hh;
                const bool zh = hasz && hh == 0;
                float acc[32], accz;
                lookback_sum<DK, kMode>(sm, p, it, nlb, a, h, zh, gL, w0, acc, accz);
                if (it.hasA) add_own_state(lb, h, zh, acc, accz);
                // phase-B start: TMEM [S | z] = g^n0 [S_start | z_start], and
                // the bf16 [S_start | z_start] operand
                uint32_t v[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(f0 * acc[e]);
                tmem_st32(lb + TM_S + 32 * h, v);
                store_sb_half(sb, a, h, acc);
                if (zh) {
                    tmem_put_z(lb + TM_S + DV, f0 * accz);
                    store_zb(sbz, a, accz);
                }
                tmem_wait_st();
            }
        }
        fence_async_shared();
        tc_fence_before();
        named_bar_sync(BAR_E2, 128);
        if (et == 0) mbar_arrive(&sm.sb_ready);
        for (int c = it.c0; c < it.c1; ++c, ++j, ++nb) {
            if (c + 1 < it.c1) {
                // state epilogue: [S | z] of chunk c+1 as the bf16 operand,
                // and with decay the rescale g^n of the accumulator
                wait_bar(&sm.s_full, ns & 1, cx);
                ++ns;
                tc_fence_after();
                const int n = min(C, p.N - (c + 1) * C);
                float f = gpow(lg, n);
                if (kMode == 2) {
                    const int j1 = j + 1;
                    // the gate slot has landed with the tiles (no need to
                    // wait for the chunk's feature map)
                    wait_bar(&sm.full[j1 % L::STAGES], (j1 / L::STAGES) & 1, cx);
                    f = gate_prod(*reinterpret_cast<const GateSlot *>(
                                      smem + (j1 % L::STAGES) * L::STAGE + L::OFF_GS),
                                  n - 1, -1);
                }
#pragma unroll
                for (int hh = 0; hh < SM::NH; ++hh) {
                    const int h = h0 + hh;
                    uint32_t v[32];
                    tmem_ld32(lb + TM_S + 32 * h, v);
                    tmem_wait_ld();
                    reg_fence(v);
                    float x[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[e] = u2f(v[e]);
                    store_sb_half(sb, a, h, x);
                    if (kMode) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(f * x[e]);
                        tmem_st32(lb + TM_S + 32 * h, v);
                    }
                }
                if (hasz) {
                    uint32_t zr = tmem_ld1(lb + TM_S + DV);
                    tmem_wait_ld();
                    reg_fence(zr);
                    const float z = u2f(zr);
                    store_zb(sbz, a, z);
                    if (kMode) tmem_put_z(lb + TM_S + DV, f * z);
                }
                if (kMode) tmem_wait_st();
                fence_async_shared();
                tc_fence_before();
                named_bar_sync(BAR_E2, 128);
                if (et == 0) mbar_arrive(&sm.sb_ready);
            }
            output_chunk<DK, kMode>(sm, p, cx, lb, row, et, it, c, j, nb);
        }
        if (p.S_out && it.seg == p.nseg - 1) {
            // the state after the sequence's last token (a decode continues
            // from it): this item's 64 value columns of S, and z once
            wait_bar(&sm.s_full, ns & 1, cx);
            ++ns;
            tc_fence_after();
#pragma unroll 1
            for (int hh = 0; hh < SM::NH; ++hh) {
                const int h = h0 + hh;
                uint32_t v[32];
                tmem_ld32(lb + TM_S + 32 * h, v);
                tmem_wait_ld();
                reg_fence(v);
                float4 *dst = reinterpret_cast<float4 *>(
                    p.S_out + ((size_t)it.bh * DK + a) * DK + 64 * it.half + 32 * h);
                const bool oks = LA_DCHECK(p.status, it.bh < p.BH && a < DK &&
                                                         64 * it.half + 32 * h + 32 <= DK);
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    if (oks)
                        dst[e] = make_float4(u2f(v[4 * e]), u2f(v[4 * e + 1]),
                                             u2f(v[4 * e + 2]), u2f(v[4 * e + 3]));
            }
            if (hasz && it.half == 0) {
                uint32_t zr = tmem_ld1(lb + TM_S + DV);
                tmem_wait_ld();
                reg_fence(zr);
                if (LA_DCHECK(p.status, it.bh < p.BH && a < DK))
                    p.z_out[(size_t)it.bh * DK + a] = u2f(zr);
            }
            tc_fence_before();
            named_bar_sync(BAR_E2, 128);
            if (et == 0) mbar_arrive(&sm.sb_ready);
        }
    }
}

// ---------------------------------------------------------------- kernel

template <int DK, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
causal_kernel(const __grid_constant__ CUtensorMap tq,
              const __grid_constant__ CUtensorMap tk,
              const __grid_constant__ CUtensorMap tv, const Params p,
              const DecayArgs dk) {
    using L = Layout<DK, kMode>;
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
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.pfull[b], 1);
            mbar_init(&sm.pt_ready[b], 128);
            mbar_init(&sm.pv_done[b], 1);
            mbar_init(&sm.o_full[b], 1);
            mbar_init(&sm.o_empty[b], 128);
        }
        mbar_init(&sm.s_full, 1);
        mbar_init(&sm.sb_ready, 1);
        mbar_init(&sm.khat_ready[0], 1);
        mbar_init(&sm.khat_ready[1], 1);
        for (int r = 0; r < 2; ++r) {
            mbar_init(&sm.item_full[r], 1);
            mbar_init(&sm.item_empty[r], 4);
        }
        mbar_init(&sm.fin, 1);
        fence_mbar_init();
    }
    // constant operand blocks: the ones column of [V | 1], and the z block of
    // [S | z] (column 0 is rewritten per chunk, the rest stays zero)
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
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the workspace clear before this kernel has completed (dependent launch)
    grid_dep_wait();
    const uint32_t tmem = sm.tmem_base;

    if (warp == 0) {
        if (lane == 0) producer<DK, kMode>(smem, sm, p, cx, &tq, &tk, &tv);
    } else if (warp == 1) {
        if (lane == 0) mma_issuer<DK, kMode>(smem, sm, p, cx, dk, tmem);
    } else if (warp < kWarpE1) {
        transform<DK, kMode>(smem, sm, p, cx, dk);
    } else if (warp < kWarpE2) {
        score_epilogue<DK, kMode>(smem, sm, p, cx, dk, tmem);
    } else {
        output_state<DK, kMode>(smem, sm, p, cx, dk, tmem);
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, TM_COLS);
}

// Automatic segment length.  Without decay: the wave rule (per-item
// overhead about three chunk times, measured).  With decay the per-chunk
// time grows once a wave's phase-A loads of K and V no longer stay in L2
// until phase B re-reads them, so segments stay short: about three items
// per SM, 2..8 chunks.
template <bool kWeighted>
int auto_segment_chunks(long long heads, int nchunks, int sms) {
    if (!kWeighted) return tchost::wave_segment_chunks(heads, nchunks, sms, 3);
    const long long units = heads * nchunks;
    const long long want = (units + 3LL * sms - 1) / (3LL * sms);
    return (int)(want < 2 ? 2 : (want > 8 ? 8 : want));
}

// With a per-head decay every head of which folds its weights (elu + 1 map,
// g >= 0.77), a chunk costs about what it costs without decay, so segments
// follow the undecayed rule (B4 H16 N4096 d64 with the decay schedule: 81.4
// us at 5-chunk segments, 71.2 us at 16).
inline bool decay_folds(const FwdShape &sh, const DecayArgs &dk) {
    if (!dk.has || !sh.phi) return false;
    for (int h = 0; h < dk.H; ++h)
        if (!(log2f(dk.g[h]) >= kFoldLog2)) return false;
    return true;
}

template <int DK, int kMode>
constexpr size_t smem_bytes() {
    return (size_t)Layout<DK, kMode>::OFF_SMALL + sizeof(Small) + 1024;
}

static_assert(smem_bytes<64, true>() <= 232448, "shared memory budget");
static_assert(smem_bytes<64, false>() <= 232448, "shared memory budget");
static_assert(smem_bytes<128, 2>() <= 232448, "shared memory budget");
static_assert(smem_bytes<64, 2>() <= 232448, "shared memory budget");

}  // namespace causal_tc

namespace {

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Work decomposition and workspace layout of one causal launch.
struct CausalPlan {
    int seg_chunks, seg0, nseg, nchunks, nhalf;
    long long items;
    size_t off_flags, off_agg, off_gprod, off_slots, total;
};

template <int DK, int kMode>
CausalPlan plan_causal(const FwdShape &sh, int seg_chunks, int sms, bool folds = false) {
    using namespace causal_tc;
    using L = Layout<DK, kMode>;
    CausalPlan pl{};
    pl.nchunks = (sh.N + C - 1) / C;
    pl.nhalf = DK / DV;
    const bool automatic = seg_chunks <= 0;
    // The gated mode follows the undecayed rule too, whether its chunks fold
    // or not (B4 H16 N4096 d64, gates uniform in [0.9, 1): 71.3 us at 5-chunk
    // segments, 62.6 us at 19 + 13; in [0.5, 1), where no chunk folds: 78.3
    // and 71.2 us; in [0.99, 1): 71.2 and 63.0 us).
    if (automatic)
        seg_chunks = (folds || kMode == 2)
                         ? auto_segment_chunks<false>(sh.BH() * pl.nhalf, pl.nchunks, sms)
                         : auto_segment_chunks<kMode != 0>(sh.BH() * pl.nhalf, pl.nchunks, sms);
    if (seg_chunks > pl.nchunks) seg_chunks = pl.nchunks;
    int seg0 = seg_chunks;
    // Two segments per head: segment 0 runs phase B from the start while
    // segment 1 first reduces segment 0's chunks (phase A, about 0.42 of a
    // phase-B chunk's time), so segment 0 takes three fifths of the chunks
    // (B4 H16 N4096 d64: 19 of 32 chunks, 50.7 us a step; 21: 52.7 us; 22:
    // 54.8 us; equal halves with segment 0 running a phase A: 56.5 us).
    if (automatic && (pl.nchunks + seg_chunks - 1) / seg_chunks == 2) {
        seg0 = 3 * pl.nchunks / 5;
        seg_chunks = pl.nchunks - seg0;
    }
    pl.seg0 = seg0;
    pl.seg_chunks = seg_chunks;
    pl.nseg = pl.nchunks <= seg0 ? 1 : 1 + (pl.nchunks - seg0 + seg_chunks - 1) / seg_chunks;
    pl.items = sh.BH() * pl.nseg * pl.nhalf;
    // workspace: control words, flags, published states
    pl.off_flags = 256;
    pl.off_agg = align_up(pl.off_flags + sizeof(int) * (size_t)pl.items, 256);
    const size_t state_bytes = (pl.nseg > 1) ? sizeof(float) * L::STATE * (size_t)pl.items : 0;
    pl.off_gprod = align_up(pl.off_agg + state_bytes, 256);
    // mode 2: the gate slots of every chunk of every head
    pl.off_slots = align_up(pl.off_gprod + (kMode == 2 ? sizeof(float) * (size_t)pl.items : 0), 256);
    pl.total = pl.off_slots +
               (kMode == 2 ? (size_t)kGateSlotBytes * (size_t)sh.BH() * (size_t)pl.nchunks : 0);
    return pl;
}

template <int DK, int kMode>
TcResult launch_causal_t(const void *q, const void *k, const void *v, void *out,
                         const FwdShape &sh, const DecayArgs &dk, int seg_chunks,
                         int *status, void *ws_in, size_t ws_bytes, float *S_out,
                         float *z_out, const float *gates, cudaStream_t stream) {
    using namespace causal_tc;
    const int BH = (int)sh.BH(), N = sh.N;
    CUtensorMap tq, tk, tv;
    cudaError_t e;
    if ((e = tchost::make_seq_map(&tq, q, BH, N, DK, C)) != cudaSuccess ||
        (e = tchost::make_seq_map(&tk, k, BH, N, DK, C)) != cudaSuccess ||
        (e = tchost::make_seq_map(&tv, v, BH, N, DK, C)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward: TMA descriptor"};
    int sms = 0;
    if ((e = tchost::sm_count(&sms)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward: device query"};
    const CausalPlan pl = plan_causal<DK, kMode>(sh, seg_chunks, sms, decay_folds(sh, dk));
    if (pl.items > (1LL << 30))
        return {LA_ERR_UNSUPPORTED, cudaSuccess, "la_forward: too many work items"};

    Params p{};
    p.BH = BH;
    p.H = sh.H;
    p.N = N;
    p.nchunks = pl.nchunks;
    p.nhalf = pl.nhalf;
    p.seg_chunks = pl.seg_chunks;
    p.seg0 = pl.seg0;
    p.nseg = pl.nseg;
    p.items = (int)pl.items;
    p.timeout = 1LL << 32;
    p.S_out = S_out;
    p.z_out = z_out;
    p.phi = sh.phi;
    p.norm = sh.norm;
    p.gates = gates;

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
    p.flags = reinterpret_cast<int *>(w8 + pl.off_flags);
    p.agg = reinterpret_cast<float *>(w8 + pl.off_agg);
    p.gprod = reinterpret_cast<float *>(w8 + pl.off_gprod);
    p.slots = reinterpret_cast<const uint8_t *>(w8 + pl.off_slots);
    p.status = status;
    p.out = static_cast<uint16_t *>(out);
    // the ticket counter, abort flag and segment flags start at zero (cleared
    // by the gate-slot kernel in the gated mode); the states need no clearing
    if (kMode == 2) {
        gate_slots_kernel<<<(unsigned)(sh.BH() * pl.nchunks), C, 0, stream>>>(
            gates, N, pl.nchunks, reinterpret_cast<GateSlot *>(w8 + pl.off_slots),
            static_cast<uint4 *>(ws), pl.off_agg / 16);
        e = cudaGetLastError();
    } else {
        e = tc_zero_words(ws, pl.off_agg, stream);
    }
    if (e == cudaSuccess) {
        const size_t smem = smem_bytes<DK, kMode>();
        auto kern = causal_kernel<DK, kMode>;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e == cudaSuccess) {
            const int grid = (int)(pl.items < sms ? pl.items : sms);
            e = tchost::launch_dependent(kern, (unsigned)grid, kThreads, smem, stream, tq, tk,
                                         tv, p, dk);
            if (e == cudaSuccess) e = cudaGetLastError();
        }
    }
    cudaError_t ef = ws_in ? cudaSuccess : cudaFreeAsync(ws, stream);
    if (e != cudaSuccess) return {LA_ERR_CUDA, e, "la_forward: causal kernel launch"};
    if (ef != cudaSuccess) return {LA_ERR_CUDA, ef, "la_forward: workspace free"};
    note_launches(2);  // workspace clear (with the gate slots when gated) + forward
    return {LA_OK, cudaSuccess, ""};
}

}  // namespace

TcResult launch_causal_tc(const void *q, const void *k, const void *v,
                          void *out, const FwdShape &sh, const DecayArgs &dk,
                          int seg_chunks, int *status, void *ws, size_t ws_bytes,
                          float *S_out, float *z_out, const float *gates,
                          cudaStream_t stream) {
    if (gates)
        return sh.d == 128
                   ? launch_causal_t<128, 2>(q, k, v, out, sh, dk, seg_chunks, status, ws, ws_bytes, S_out, z_out, gates, stream)
                   : launch_causal_t<64, 2>(q, k, v, out, sh, dk, seg_chunks, status, ws, ws_bytes, S_out, z_out, gates, stream);
    // d = 128 without gates: one CTA per (head, segment) over all 128 value
    // columns (la_causal_wide.cu)
    if (sh.d == 128)
        return launch_causal_wide(q, k, v, out, sh, dk, seg_chunks, status, ws, ws_bytes,
                                  S_out, z_out, stream);
    return dk.has ? launch_causal_t<64, true>(q, k, v, out, sh, dk, seg_chunks, status, ws, ws_bytes, S_out, z_out, nullptr, stream)
                  : launch_causal_t<64, false>(q, k, v, out, sh, dk, seg_chunks, status, ws, ws_bytes, S_out, z_out, nullptr, stream);
}

size_t causal_tc_workspace_bytes(const FwdShape &sh, bool decay, int seg_chunks, int sms) {
    if (sh.d == 128) return causal_wide_workspace_bytes(sh, seg_chunks, sms);
    if (!decay) return plan_causal<64, false>(sh, seg_chunks, sms).total;
    // the decay values are not known here: cover both segment rules
    const size_t a = plan_causal<64, true>(sh, seg_chunks, sms, false).total;
    const size_t b = plan_causal<64, true>(sh, seg_chunks, sms, true).total;
    return a > b ? a : b;
}

}  // namespace la

// ============================================================================
// Allocation-free variant of the causal tensor-core forward.
//
// Some callers cannot allocate device memory at the point where they run
// attention: code recorded into a CUDA graph whose capture mode forbids
// allocation nodes, hosts that reserve all device memory up front (embedded
// and real-time deployments, memory-pool-managed servers), and plug-in or
// interop layers that are handed input and output buffers by a host
// framework and must not own allocations of their own.  For them
// la_forward_causal_noalloc runs the same chunkwise causal kernel, but its
// workspace (ticket counter, segment flags and published segment states)
// lives in the fixed device array below instead of a cudaMallocAsync block.
//
// The array is LA_NOALLOC_SCRATCH_BYTES (16 MiB) and every GPU that loads
// this library's causal kernels keeps it until the process exits.  Requests
// are fitted into it by lengthening the sequence segments; a request whose
// workspace does not fit even with one segment per head is rejected.
// ============================================================================

static __device__ __align__(256) unsigned char
    la_noalloc_scratch[LA_NOALLOC_SCRATCH_BYTES];

namespace la {
namespace {

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[64] = {};

// Device address of la_noalloc_scratch on the current device.  The symbol's
// name is only a host-side stand-in, so the address is looked up once per
// device (with that device current) and cached.
cudaError_t noalloc_scratch(char **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, la_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_noalloc_ptr[dev] = p;
    }
    *out = static_cast<char *>(g_noalloc_ptr[dev]);
    return cudaSuccess;
}

template <int DK, int kMode>
TcResult launch_causal_noalloc_t(const void *q, const void *k, const void *v,
                                 void *out, const FwdShape &sh,
                                 const DecayArgs &dk, int *status,
                                 cudaStream_t stream) {
    using namespace causal_tc;
    using L = Layout<DK, kMode>;
    const int BH = (int)sh.BH(), N = sh.N;
    CUtensorMap tq, tk, tv;
    cudaError_t e;
    if ((e = tchost::make_seq_map(&tq, q, BH, N, DK, C)) != cudaSuccess ||
        (e = tchost::make_seq_map(&tk, k, BH, N, DK, C)) != cudaSuccess ||
        (e = tchost::make_seq_map(&tv, v, BH, N, DK, C)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward_causal_noalloc: TMA descriptor"};
    int sms = 0;
    if ((e = tchost::sm_count(&sms)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward_causal_noalloc: device query"};
    char *scratch = nullptr;
    if ((e = noalloc_scratch(&scratch)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward_causal_noalloc: scratch address"};

    Params p{};
    p.BH = BH;
    p.H = sh.H;
    p.N = N;
    p.nchunks = (N + C - 1) / C;
    p.nhalf = DK / DV;
    int seg = decay_folds(sh, dk) ? auto_segment_chunks<false>(BH * p.nhalf, p.nchunks, sms)
                                  : auto_segment_chunks<kMode != 0>(BH * p.nhalf, p.nchunks, sms);
    // lengthen segments until the workspace fits the static scratch
    size_t off_agg = 0, total = 0;
    long long items = 0;
    for (;;) {
        const int nseg = (p.nchunks + seg - 1) / seg;
        items = (long long)BH * nseg * p.nhalf;
        off_agg = align_up(256 + sizeof(int) * (size_t)items, 256);
        const size_t sb = nseg > 1 ? sizeof(float) * L::STATE * (size_t)items : 0;
        total = off_agg + sb;
        if (total <= (size_t)LA_NOALLOC_SCRATCH_BYTES || seg >= p.nchunks) break;
        seg = seg * 2 < p.nchunks ? seg * 2 : p.nchunks;
    }
    if (total > (size_t)LA_NOALLOC_SCRATCH_BYTES || items > (1LL << 30))
        return {LA_ERR_UNSUPPORTED, cudaSuccess,
                "la_forward_causal_noalloc: the problem needs more workspace "
                "than the 16 MiB static scratch holds (too many heads)"};
    p.seg_chunks = seg;
    p.seg0 = seg;
    p.nseg = (p.nchunks + seg - 1) / seg;
    p.items = (int)items;
    p.timeout = 1LL << 32;
    p.phi = 1;
    p.norm = 1;
    p.ctrl = reinterpret_cast<int *>(scratch);
    p.flags = reinterpret_cast<int *>(scratch + 256);
    p.agg = reinterpret_cast<float *>(scratch + off_agg);
    p.status = status;
    p.out = static_cast<uint16_t *>(out);
    // the counter and flags must start at zero; the states need no clearing
    if ((e = tc_zero_words(scratch, off_agg, stream)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward_causal_noalloc: clearing flags"};
    const size_t smem = smem_bytes<DK, kMode>();
    auto kern = causal_kernel<DK, kMode>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward_causal_noalloc: kernel attribute"};
    const int grid = (int)(items < sms ? items : sms);
    e = tchost::launch_dependent(kern, (unsigned)grid, kThreads, smem, stream, tq, tk, tv, p,
                                 dk);
    if (e != cudaSuccess || (e = cudaGetLastError()) != cudaSuccess)
        return {LA_ERR_CUDA, e, "la_forward_causal_noalloc: kernel launch"};
    note_launches(2);  // flag clear + forward
    return {LA_OK, cudaSuccess, ""};
}

la_status noalloc_fail(la_status s, const char *msg) {
    set_last_error(msg);
    return s;
}

}  // namespace
}  // namespace la

extern "C" __attribute__((visibility("default")))
la_status la_forward_causal_noalloc(const void *q, const void *k,
                                    const void *v, void *out, int B, int H,
                                    int N, int d, const float *decay,
                                    la_stream_t stream) {
    using namespace la;
    if (!q || !k || !v || !out)
        return noalloc_fail(LA_ERR_INVALID_ARG,
                            "la_forward_causal_noalloc: null tensor pointer");
    if (B < 0 || H < 0 || N < 0)
        return noalloc_fail(LA_ERR_INVALID_ARG,
                            "la_forward_causal_noalloc: negative B, H or N");
    if (d != 64 && d != 128)
        return noalloc_fail(LA_ERR_UNSUPPORTED,
                            "la_forward_causal_noalloc: d must be 64 or 128");
    if (out == q || out == k || out == v)
        return noalloc_fail(LA_ERR_INVALID_ARG,
                            "la_forward_causal_noalloc: out aliases an input");
    const uintptr_t mis = (reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                           reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out)) & 15u;
    if (mis)
        return noalloc_fail(LA_ERR_UNSUPPORTED,
                            "la_forward_causal_noalloc: tensors must be 16-byte aligned");
    DecayArgs dk;
    dk.has = 0;
    dk.H = H > 0 ? H : 1;
    if (decay) {
        if (H > LA_MAX_DECAY_HEADS)
            return noalloc_fail(LA_ERR_UNSUPPORTED,
                                "la_forward_causal_noalloc: decay given for more than 1024 heads");
        for (int h = 0; h < H; ++h) {
            const float g = decay[h];
            if (!(g >= 0.f && g <= 1.f))
                return noalloc_fail(LA_ERR_INVALID_ARG,
                                    "la_forward_causal_noalloc: decay values must lie in [0, 1]");
            dk.g[h] = g;
        }
        dk.has = 1;
    }
    const FwdShape sh{B, H, N, d};
    if (sh.BH() == 0 || N == 0) return LA_OK;
    if (sh.BH() > 2147483647LL || (long long)N * d > (1LL << 40))
        return noalloc_fail(LA_ERR_UNSUPPORTED,
                            "la_forward_causal_noalloc: problem too large");
    cudaError_t ce;
    int *status = device_status_word(&ce);
    if (!status) {
        set_last_error("la_forward_causal_noalloc: status word lookup failed");
        return LA_ERR_CUDA;
    }
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    TcResult r;
    if (d == 128) {
        char *scratch = nullptr;
        const cudaError_t e = noalloc_scratch(&scratch);
        r = e != cudaSuccess
                ? TcResult{LA_ERR_CUDA, e, "la_forward_causal_noalloc: scratch address"}
                : launch_causal_wide_fixed(q, k, v, out, sh, dk, status, scratch,
                                           (size_t)LA_NOALLOC_SCRATCH_BYTES, s);
    } else
        r = dk.has ? launch_causal_noalloc_t<64, true>(q, k, v, out, sh, dk, status, s)
                   : launch_causal_noalloc_t<64, false>(q, k, v, out, sh, dk, status, s);
    if (r.status != LA_OK) {
        char msg[256];
        if (r.status == LA_ERR_CUDA)
            std::snprintf(msg, sizeof(msg), "%s: %s", r.where, cudaGetErrorString(r.cuda));
        else
            std::snprintf(msg, sizeof(msg), "%s", r.where);
        set_last_error(msg);
    }
    return r.status;
}
