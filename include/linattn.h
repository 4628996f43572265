/*
 * linattn.h -- C ABI of the GB300 (sm_103a) kernelised linear-attention
 * library (liblinattn.so).
 *
 * The operation ("Linear Attention", generalised-kernel equations and the
 * causal running statistics; "Story of Attention - Part 5: Linear Attention:
 * Kernels, Decay, and Gating", section 1a):
 *
 *   phi(x)  = elu(x) + 1   (alpha = 1), applied elementwise to q and k only
 *   non-causal   y_i = phi(q_i)^T [sum_j phi(k_j) v_j^T] / phi(q_i)^T [sum_j phi(k_j)]
 *   causal       S_t = g S_{t-1} + phi(k_t) v_t^T,  z_t = g z_{t-1} + phi(k_t),
 *                y_t = phi(q_t)^T S_t / phi(q_t)^T z_t      (update, then read)
 *
 * with an optional per-head scalar decay g ("Linear Attention: Removing the
 * Softmax Buys Associativity", the forget-gate passage; Part 5, section 4
 * recurrent form), g = 1 when no decay is given.  There is no 1/sqrt(d)
 * scaling and no epsilon in the denominator (phi > 0 makes it positive).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller (except
 *     la_forward_host's, which are host pointers); the library never frees
 *     or retains them after the call is enqueued.
 *   - Sequences are row-major contiguous [B][H][N][d] (d fastest); decode
 *     inputs are [B][H][d]; states S are [B][H][d][d] with S[a][c],
 *     a = key-feature index, c = value index; normalisers z are [B][H][d].
 *   - q, k, v and out share one dtype (`dtype`); outputs are rounded to it
 *     with round-to-nearest-even.  Accumulation is always fp32.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the
 *     legacy default stream) and performs no implicit synchronisation.
 *     Arguments are validated on the host before anything is enqueued; a
 *     rejected call enqueues nothing.
 *   - Calls are thread-safe.  The library's only global mutable state is a
 *     per-device status word written by kernels that detect a device-side
 *     problem (a bounded wait that ran out); read it with
 *     la_check_device_status().
 */
#ifndef LINATTN_H
#define LINATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same underlying type as cudaStream_t, so that a cudaStream_t (or
 * torch.cuda.Stream.cuda_stream) can be passed directly. */
typedef struct CUstream_st *la_stream_t;

typedef enum {
    LA_OK = 0,
    LA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, bad decay, ...      */
    LA_ERR_UNSUPPORTED = 2,  /* valid request this build cannot run          */
    LA_ERR_CUDA = 3,         /* a CUDA runtime call or launch failed         */
    LA_ERR_NO_MEMORY = 4,    /* workspace allocation failed                  */
    LA_ERR_TIMEOUT = 5,      /* a device-side bounded wait gave up           */
    LA_ERR_INTERNAL = 6      /* a debug build's device-side index check failed */
} la_status;

typedef enum { LA_F32 = 0, LA_BF16 = 1 } la_dtype;

/* Method variant for la_forward_variant / la_decode_step_variant. */
typedef enum { LA_PHI_ELU1 = 0, LA_PHI_IDENTITY = 1 } la_feature_map;
typedef struct {
    int feature_map; /* LA_PHI_ELU1: phi(x) = elu(x) + 1 (the default);
                        LA_PHI_IDENTITY: phi(x) = x                         */
    int normalise;   /* 1: divide by phi(q)^T z (the default); 0: no
                        denominator                                         */
} la_variant;

/* Largest head dimension accepted by any entry point. */
#define LA_MAX_D 256
/* Largest number of heads for which a per-head decay can be given. */
#define LA_MAX_DECAY_HEADS 1024

/*
 * la_forward -- full-sequence linear attention.
 *
 * Defined by the non-causal form phi(Q)[phi(K)^T V] / phi(Q)[phi(K)^T 1]
 * ("Story of Attention - Part 5", section 1a, matrix form) when causal == 0,
 * and by the causal running-state recurrence (same section, causal form;
 * "Linear Attention", cumulative running statistics) when causal == 1.
 *
 *   q, k, v  [B][H][N][d] device, dtype `dtype`, read only.
 *   out      [B][H][N][d] device, dtype `dtype`, written; may not alias
 *            q, k or v.
 *   B, H, N  >= 0 (B*H*N == 0 is a no-op returning LA_OK, and then q, k,
 *            v, out may be NULL); d in 1..LA_MAX_D.
 *   causal   0 or 1.
 *   decay    HOST array of H floats g_h in [0, 1] (read during the call, not
 *            retained), or NULL for g = 1.  Only valid with causal == 1:
 *            the pages define decay for the recurrence only, so a decay with
 *            causal == 0 is LA_ERR_INVALID_ARG.
 *   dtype    LA_F32 or LA_BF16.  fp32 inputs run on the fp32 CUDA-core path
 *            (no TF32); bf16 inputs with d in {64, 128} run on the tcgen05
 *            tensor-core kernels, other d on the CUDA-core path.
 *
 * Workspace: the tensor-core kernels, and the CUDA-core kernels when they
 * cut a sequence into segments (or reduce a non-causal state), need a small
 * stream-ordered scratch (per-segment states and flags), allocated with
 * cudaMallocAsync on `stream` and freed with cudaFreeAsync on the same
 * stream; LA_ERR_NO_MEMORY if that fails.
 */
la_status la_forward(const void *q, const void *k, const void *v, void *out,
                     int B, int H, int N, int d, int causal,
                     const float *decay, la_dtype dtype, la_stream_t stream);

/*
 * la_forward_ex -- la_forward with explicit kernel selection, for tests and
 * measurement.  `path`: 0 = automatic (what la_forward does), 1 = force the
 * fp32 CUDA-core kernels (any dtype), 2 = force the tensor-core kernels
 * (LA_ERR_UNSUPPORTED where they do not apply).  `segment_chunks`: 0 =
 * automatic, else the number of chunks per sequence segment that one CTA
 * takes (sequence parallelism inside a head; chunks of 128 tokens on the
 * tensor cores, of 32 on the CUDA cores).
 */
la_status la_forward_ex(const void *q, const void *k, const void *v,
                        void *out, int B, int H, int N, int d, int causal,
                        const float *decay, la_dtype dtype, int path,
                        int segment_chunks, la_stream_t stream);

/*
 * la_forward_host -- la_forward on HOST buffers (the one entry point whose
 * tensors are host pointers).  The pages define only the operation (as for
 * la_forward); moving the data to and from the GPU has no counterpart there.
 * The call copies q, k, v to a caller-provided device workspace, runs the
 * forward there and copies out back, split into at most 4 groups of heads so
 * that the host-to-device copy of one group, the kernels of the one before
 * and the device-to-host copy of the one before that overlap (two copy
 * streams owned by the library, one per direction, created on first use).
 *
 *   q, k, v   [B][H][N][d] host, dtype `dtype`, read only.  Page-locked
 *             memory (cudaHostAlloc, cudaHostRegister, torch pin_memory)
 *             gives asynchronous full-speed copies; pageable memory works,
 *             but the CUDA driver stages its copies and the call then blocks.
 *   out       [B][H][N][d] host, written; may not alias q, k or v.
 *   B, H, N, d, causal, decay, dtype   as la_forward (decay is a host
 *             array of H floats, read during the call).
 *   workspace device buffer, 256-byte aligned, of at least
 *             la_forward_host_workspace_bytes(B, H, N, d, dtype) bytes,
 *             owned by the caller; it holds the device copies of q, k, v and
 *             out and must not be used by anything else until `stream` has
 *             passed the call.
 *   stream    the copies start after the work already enqueued on `stream`;
 *             `stream` continues only after the last output copy, so out is
 *             complete once `stream` reaches work enqueued after the call
 *             (e.g. cudaStreamSynchronize(stream)).
 *
 * Errors: validation as la_forward (LA_ERR_INVALID_ARG also for a missing,
 * unaligned or too small workspace); a failure part-way through returns its
 * status with `stream` still ordered after the copies already enqueued, and
 * out unspecified.  Calls on one device are serialised on the host while
 * they enqueue (the copy streams and their events are shared).
 */
la_status la_forward_host(const void *q, const void *k, const void *v,
                          void *out, int B, int H, int N, int d, int causal,
                          const float *decay, la_dtype dtype, void *workspace,
                          size_t workspace_bytes, la_stream_t stream);

/* Device workspace bytes la_forward_host needs for this problem (0 for an
 * invalid shape or dtype). */
size_t la_forward_host_workspace_bytes(int B, int H, int N, int d,
                                       la_dtype dtype);

/*
 * la_decode_step -- one recurrent decode step per head: with
 * phi_k = phi(k), S <- S + phi_k v^T, z <- z + phi_k, then
 * out = phi(q)^T S / phi(q)^T z  (update, then read; "Linear Attention",
 * running statistics and per-token inference cost O(d^2) arithmetic and
 * O(d^2) memory, independent of history).
 *
 *   S        [B][H][d][d] fp32 device, read and written in place.
 *   z        [B][H][d]    fp32 device, read and written in place.
 *   q, k, v  [B][H][d] device, dtype `dtype`, read only.
 *   out      [B][H][d] device, dtype `dtype`, written.
 *   B, H >= 0 (B*H == 0 is a no-op), d in 1..LA_MAX_D.
 * The caller owns the recurrent state; saving and restoring S and z is how
 * a decode is checkpointed and resumed.
 */
la_status la_decode_step(float *S, float *z, const void *q, const void *k,
                         const void *v, void *out, int B, int H, int d,
                         la_dtype dtype, la_stream_t stream);

/*
 * la_decode_step_ex -- la_decode_step with a per-head decay g:
 * S <- g S + phi_k v^T, z <- g z + phi_k, then out = phi(q)^T S / phi(q)^T z
 * (the recurrence with the forget-gate passage's scalar g; "Story of
 * Attention - Part 5", section 4, recurrent form S_t = g S_{t-1} + k_t v_t^T).
 *   decay    HOST array of H floats in [0, 1] (read during the call), or NULL
 *            for g = 1 (then identical to la_decode_step).
 * Other arguments, layouts and errors as la_decode_step; LA_ERR_UNSUPPORTED
 * for a decay over more than LA_MAX_DECAY_HEADS heads.
 */
la_status la_decode_step_ex(float *S, float *z, const void *q, const void *k,
                            const void *v, void *out, int B, int H, int d,
                            const float *decay, la_dtype dtype,
                            la_stream_t stream);

/*
 * la_forward_causal_state -- the causal form of la_forward that also returns
 * the final state: S_N = sum_t g^(N-1-t) phi(k_t) v_t^T and z_N likewise,
 * i.e. the running statistics after the last token ("Linear Attention",
 * running statistics; the state an RNN-style decode continues from).  It is
 * the prefill half of a prefill -> decode hand-off: la_decode_step(_ex) on S
 * and z then continues the same sequences.
 *   q, k, v, out, B, H, N, d, decay, dtype   as la_forward with causal = 1.
 *   S        [B][H][d][d] fp32 device, written (S[a][c]: a key feature, c
 *            value column; the layout la_decode_step reads); 16-byte aligned.
 *   z        [B][H][d] fp32 device, written.
 * N == 0 writes the zero state.  Errors as la_forward, plus
 * LA_ERR_INVALID_ARG for a NULL or unaligned S or a NULL z.
 */
la_status la_forward_causal_state(const void *q, const void *k, const void *v,
                                  void *out, float *S, float *z, int B, int H,
                                  int N, int d, const float *decay,
                                  la_dtype dtype, la_stream_t stream);

/*
 * la_forward_variant / la_decode_step_variant -- la_forward_ex (automatic
 * kernel and segment choice) and la_decode_step_ex with the feature map and
 * the normaliser selectable.  With {LA_PHI_IDENTITY, 0} and a decay this is
 * retention ("Story of Attention - Part 5", section 4: recurrent form
 * S_t = g S_{t-1} + k_t v_t^T, o_t = q_t S_t; parallel form (Q K^T (.) D) V
 * with D_ij = g^(i-j) for i >= j); with {LA_PHI_ELU1, 0} linear attention
 * without the denominator.
 *   variant  NULL for {LA_PHI_ELU1, 1} (then identical to la_forward_ex /
 *            la_decode_step_ex); LA_ERR_INVALID_ARG for a feature_map other
 *            than the two above or a normalise other than 0 or 1.
 * Without the normaliser z is still carried (and, for the decode step,
 * updated) but not used.  Other arguments and errors as la_forward and
 * la_decode_step_ex.
 */
la_status la_forward_variant(const void *q, const void *k, const void *v,
                             void *out, int B, int H, int N, int d, int causal,
                             const float *decay, la_dtype dtype,
                             const la_variant *variant, la_stream_t stream);
la_status la_decode_step_variant(float *S, float *z, const void *q,
                                 const void *k, const void *v, void *out, int B,
                                 int H, int d, const float *decay,
                                 la_dtype dtype, const la_variant *variant,
                                 la_stream_t stream);

/*
 * la_forward_gated / la_decode_step_gated -- the causal recurrence with a
 * data-dependent scalar gate per token and head instead of a fixed decay:
 * S_t = alpha_t S_{t-1} + phi(k_t) v_t^T, z_t = alpha_t z_{t-1} + phi(k_t),
 * y_t = phi(q_t)^T S_t / phi(q_t)^T z_t ("Linear Attention", GLA's
 * S_t = G_t (.) S_{t-1} + k_t v_t^T with G_t = alpha_t, the scalar forget
 * gate alpha_t of "Story of Attention - Part 5", section 7).
 *   gates    DEVICE fp32, [B][H][N] for la_forward_gated (alpha of every
 *            token) or [B][H] for la_decode_step_gated (alpha of this step's
 *            token), values in [0, 1].  The values are not checked (they live
 *            on the device); outside [0, 1] the results are unspecified.
 *   variant  as la_forward_variant (NULL: elu(x) + 1 with the normaliser).
 * Other arguments as la_forward (causal) and la_decode_step.  The forward
 * runs where la_forward would (bf16 with d in {64, 128}: the tcgen05
 * kernels; otherwise the fp32 CUDA-core kernels); the decode step is the
 * same kernel as la_decode_step.
 */
la_status la_forward_gated(const void *q, const void *k, const void *v,
                           void *out, const float *gates, int B, int H, int N,
                           int d, la_dtype dtype, const la_variant *variant,
                           la_stream_t stream);
la_status la_decode_step_gated(float *S, float *z, const void *q, const void *k,
                               const void *v, void *out, const float *gates,
                               int B, int H, int d, la_dtype dtype,
                               const la_variant *variant, la_stream_t stream);

/*
 * la_decode_step_delta -- one delta-rule decode step per head ("Story of
 * Attention - Part 5", section 7, Gated DeltaNet / Delta Attention: one step
 * of online gradient descent on 1/2 ||S_{t-1} k_t - v_t||^2, with the scalar
 * forget gate alpha_t):
 *   S_t = alpha S_{t-1} + beta (v_t - alpha S_{t-1} k_t) k_t^T,  o_t = S_t q_t
 * in the page's orientation, where S k is the value stored for key k.  No
 * feature map and no normaliser (the page's form; a model normalises k).
 *   S        [B][H][d][d] fp32 device, read and written in place, stored as
 *            in la_decode_step: S[a][c] with a the key feature and c the
 *            value column (the transpose of the page's S).
 *   q, k, v  [B][H][d] device, dtype `dtype`, read only.
 *   out      [B][H][d] device, dtype `dtype`, written.
 *   beta     DEVICE fp32 [B][H]: this step's update strength per head.
 *   alpha    DEVICE fp32 [B][H]: this step's forget gate per head, or NULL
 *            for alpha = 1 (plain DeltaNet).  beta and alpha are not checked
 *            (the page's ranges are beta in [0, 1], alpha in (0, 1)).
 *   B, H >= 0 (B*H == 0 is a no-op), d in 1..LA_MAX_D.
 */
la_status la_decode_step_delta(float *S, const void *q, const void *k,
                               const void *v, void *out, const float *beta,
                               const float *alpha, int B, int H, int d,
                               la_dtype dtype, la_stream_t stream);

/*
 * la_forward_delta -- the delta rule of la_decode_step_delta over whole
 * sequences ("Story of Attention - Part 5", section 7): for t = 1..N,
 *   S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T,
 *   o_t = S_t q_t,
 * with one beta and one alpha per token and head.  The pages name a
 * chunkwise form of this rule but do not give it; this is the recurrent form
 * on CUDA cores in fp32 (value columns of a head in parallel, tokens in order).
 *   q, k, v  [B][H][N][d] device, dtype `dtype`, read only.
 *   out      [B][H][N][d] device, dtype `dtype`, written (o_t).
 *   beta     DEVICE fp32 [B][H][N]: each token's update strength.
 *   alpha    DEVICE fp32 [B][H][N]: each token's forget gate, or NULL for
 *            alpha = 1 (plain DeltaNet).  beta and alpha are not checked.
 *   S        DEVICE fp32 [B][H][d][d] (S[a][c], a key feature, as in
 *            la_decode_step_delta) holding the state before the first token;
 *            it receives the state after the last one, so that
 *            la_decode_step_delta continues the sequences.  NULL: start from
 *            zero and return no state.
 *   B, H, N >= 0 (B*H*N == 0 is a no-op), d in 1..LA_MAX_D.
 */
la_status la_forward_delta(const void *q, const void *k, const void *v, void *out,
                           const float *beta, const float *alpha, float *S, int B,
                           int H, int N, int d, la_dtype dtype, la_stream_t stream);

/* Size of the fixed device scratch used by la_forward_causal_noalloc. */
#define LA_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * la_forward_causal_noalloc -- the causal form of la_forward (bf16 only),
 * for callers that cannot allocate device memory: work recorded into a CUDA
 * graph whose capture forbids allocation, hosts that reserve all device
 * memory up front, and plug-in layers that are handed their buffers and may
 * not own allocations.  The pages have no counterpart of this entry point;
 * it exists only for such callers.
 *
 * Same arguments and meaning as la_forward with causal == 1 and
 * dtype == LA_BF16: q, k, v, out are caller-owned device tensors
 * [B][H][N][d] (16-byte aligned), d must be 64 or 128, `decay` is a host
 * array of H values in [0, 1] or NULL.  It runs the same tensor-core kernel,
 * but its workspace lives in a static device array of
 * LA_NOALLOC_SCRATCH_BYTES (16 MiB) that every GPU which loads the library's
 * causal kernels keeps until the process exits.  The call makes no
 * cudaMalloc/cudaFree or other allocating call.  It enqueues two kernels on
 * `stream`: a small zeroing kernel that clears the part of the scratch that
 * must start at zero (ticket counter and segment flags), then the forward,
 * launched with programmatic stream serialisation: it may run its set-up
 * while the zeroing kernel finishes and waits for it (griddepcontrol.wait)
 * before touching memory; stream capture records a programmatic edge
 * between the two kernel nodes.
 *   - Sequence segments are lengthened until the workspace fits the
 *     scratch; if it cannot fit even with one segment per head the call
 *     returns LA_ERR_UNSUPPORTED ("needs more workspace than ...") and
 *     enqueues nothing.  Other shapes or dtypes: LA_ERR_UNSUPPORTED.
 *   - The first call on each device looks up the scratch array's device
 *     address (cudaGetSymbolAddress) with that device current; make that
 *     first call before any stream capture.
 *   - All calls on a device share the one scratch array, which keeps the
 *     last call's contents.  Calls whose kernels can overlap on the GPU
 *     (different streams without ordering between them, or several host
 *     threads) race on it and give wrong results: order them.
 */
la_status la_forward_causal_noalloc(const void *q, const void *k,
                                    const void *v, void *out, int B, int H,
                                    int N, int d, const float *decay,
                                    la_stream_t stream);

/*
 * la_check_device_status -- synchronises `stream`, then reads and clears the
 * current device's status word.  Returns LA_ERR_TIMEOUT if a kernel gave up
 * on a bounded wait since the last check (its outputs are then not valid),
 * LA_ERR_INTERNAL if, in a library built with LA_DEBUG, a device-side index
 * check failed (la_last_error names the source line), LA_ERR_CUDA if the
 * synchronisation itself failed, else LA_OK.
 */
la_status la_check_device_status(la_stream_t stream);

/* Static, human-readable name of a status code. */
const char *la_status_string(la_status s);

/* Detail of the last failed call on the calling thread ("" if none). */
const char *la_last_error(void);

/* ABI version of this header: 1. */
int la_abi_version(void);

/* Number of kernels this library has enqueued in this process (all devices,
 * all streams) since it was loaded; for measurement and launch accounting. */
unsigned long long la_kernel_launch_count(void);

/*
 * Testing hooks.  The pages have no counterpart: these exist so that the
 * library's own tests can drive its failure paths without faulting a GPU.
 * Each applies to the calling thread only and is consumed by the next call
 * it affects.
 *
 * la_debug_inject_timeout -- the next d = 128 causal tensor-core launch
 * (la_forward and friends with bf16, d = 128, no gates) bounds every wait by
 * `wait_cycles` clock cycles (>= 4096) instead of about two seconds, and
 * segment `hold_segment` of every head never publishes the state it holds
 * (-1: all publish).  Segment s >= 1 holds the local state of segment s - 1
 * and publishes it when a segment after s needs it (s = 1 .. nseg - 2;
 * segment 0 and the last segment publish nothing).  The segments after
 * `hold_segment` then wait in vain and their waits run out: the launch records
 * LA_ERR_TIMEOUT in the device status word, every later wait of the launch
 * passes through, it finishes (outputs invalid) and la_check_device_status
 * reports LA_ERR_TIMEOUT.  LA_ERR_INVALID_ARG for wait_cycles < 4096.
 *
 * la_debug_fail_next_allocs -- the next `n` stream-ordered workspace
 * allocations of the forward kernels (tensor-core launches given no
 * workspace, and CUDA-core launches over more than one segment per head, or
 * non-causal) fail: those calls return LA_ERR_NO_MEMORY and enqueue nothing.
 * n = 0 clears the hook; LA_ERR_INVALID_ARG for n < 0.
 */
la_status la_debug_inject_timeout(long long wait_cycles, int hold_segment);
la_status la_debug_fail_next_allocs(int n);

#ifdef __cplusplus
}
#endif
#endif /* LINATTN_H */
