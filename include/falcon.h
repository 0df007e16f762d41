/*
 * falcon.h — C ABI of the GB300 Falcon fast-weight forward library
 * (libfalcon.so, built for sm_103a).
 *
 * The method: a fixed-size fast-weight state S (d_k x d_v, fp32) is written
 * once per token by one normalised online gradient step on the
 * prefix-aligned pair (x_t, v_t) = (phi(k_{t-1}), v_t), with a shrinkage
 * decay gamma_t = 1 - lambda_t kept >= eps_gamma, and read after the write,
 * o_t = S_t^T q_t.  Sources, cited by page title and section:
 *   [FW]  "Falcon 家族重新对齐 fast-weight 记忆" (zhouql-dev explainer):
 *         本质 (pair alignment), Falcon 家族 (variants, knobs),
 *         三种等价形式 (recurrent / masked-parallel / chunked forms).
 *   [JC]  "给记忆装一个“及时纠错”的开关" (long write-up):
 *         把记忆更新变成一次梯度下降 (gradient step, NLMS step),
 *         Falcon家族六个变体各管一段 (1/2/3 and A variants, batched solve),
 *         数学上的稳定阀门:正衰减钳制 (decay floor eps_gamma),
 *         三种视角看同一个更新 (the three forms, WY representation).
 *
 * Update of one step t (window W(t) = existing pairs among the last W;
 * W = 1 except for Falcon-3/3A; n_t = |W(t)|; e_t = mean ||x_j||^2 over W(t)):
 *   gamma_t = clamp(1 - lambda_t, eps_gamma, 1)
 *   eta_t   = beta_t / (eps + e_t)          (scalar, or per value channel)
 *   Z       = gamma_t S_{t-1}
 *   regression (1, 2, 3):  S_t = Z + (1/n_t) sum_j x_j (eta_t * (v_j - Z^T x_j))^T
 *   additive  (1A, 2A, 3A): S_t = Z + (1/n_t) sum_j x_j (eta_t * v_j)^T
 *   o_t = S_t^T q_t
 * The pair of a token whose global index (carry pos + local index) is < 1
 * does not exist (it would need the key before the sequence) and writes
 * nothing; a step with no existing pair only decays.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library never allocates device memory.  Scratch memory, where needed,
 *     is the caller's `workspace` of at least the size the matching
 *     *_workspace_size() call returns, 256-byte aligned.
 *   - Layouts are dense row-major: q, k [B, T, H, dk]; v, o [B, T, H, dv];
 *     beta [B, T, H] (Falcon-2/2A: [B, T, H, dv]); lambda [B, T, H].
 *     q, k, v, o, carry k_prev / win_x / win_v use the params' dtype
 *     (bf16 or fp32); beta, lambda and the state S are fp32; pos is int64.
 *     q and k are the features phi(q), phi(k): the caller applies phi.
 *   - Work is enqueued asynchronously on `stream` (a cudaStream_t passed as
 *     void*; NULL = the legacy default stream).  Errors found on the host
 *     (arguments, shapes) return before anything is enqueued.
 *   - Return value: FALCON_OK (0) or a negative FALCON_ERR_* code; no
 *     exception crosses the ABI.  FALCON_ERR_CUDA reports a launch error
 *     (cudaGetLastError after the launches).
 *   - Inputs must not overlap outputs.  The chunk forward reads carry_in
 *     and writes carry_out; the two must not overlap (use two carries).
 *     The recurrent step updates its carry in place.
 */
#ifndef FALCON_H
#define FALCON_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Variants [FW Falcon 家族; JC Falcon家族六个变体各管一段]:
 * 1 scalar step, 2 per-value-channel step, 3 sliding-window mini-batch of the
 * last `window` pairs (window-averaged); "A" = inner-product objective,
 * additive write. */
typedef enum {
  FALCON_1 = 0,
  FALCON_1A = 1,
  FALCON_2 = 2,
  FALCON_2A = 3,
  FALCON_3 = 4,
  FALCON_3A = 5
} falcon_variant_t;

typedef enum { FALCON_BF16 = 0, FALCON_F32 = 1 } falcon_dtype_t;

/* Which key a value is paired with.  PREFIX (the method): pair t is
 * (phi(k_{t-1}), v_t) [FW 本质; JC 一个被忽略的时间差], x_0 the carried k_prev,
 * and a pair with global index < 1 does not exist.  SAME_STEP (the ablation
 * the pages set against it, the usual delta-rule pairing): pair t is
 * (phi(k_t), v_t), every pair with global index >= 0 exists and k_prev is
 * not read (it is still written to a carry).  Window rings hold zeros for
 * pairs that do not exist. */
typedef enum { FALCON_PAIR_PREFIX = 0, FALCON_PAIR_SAME_STEP = 1 } falcon_pairing_t;

/* Steps either side of the path, done by the library when asked
 * [FW 三种等价形式 (phi(Q), phi(K)); JC 把记忆更新变成一次梯度下降]:
 * L2NORM_QK: q and k are raw projections; the feature map phi is the
 *   per-token L2 normalisation x / max(|x|, 1e-12) (fp32, then the dtype).
 *   Carried keys (k_prev, win_x) hold features phi(k).
 * GATE_LOGITS: beta and lambda hold logits: beta = sigmoid(b) and
 *   lambda = sigmoid(a), i.e. gamma = 1 - lambda = sigmoid(-a) before the
 *   eps_gamma floor.
 * The chunk forward applies them in one pass over the inputs into its
 * workspace (falcon_workspace_size counts it), the varlen forward in its
 * gather pass, the recurrent step inside its kernel.  The backward and the
 * masked-parallel reference take features and gates (prologue must be 0). */
typedef enum {
  FALCON_PROLOGUE_L2NORM_QK = 1,
  FALCON_PROLOGUE_GATE_LOGITS = 2
} falcon_prologue_t;

/* Kernel family for the chunk forward.  AUTO picks the tensor-core path
 * (tcgen05 + TMEM + TMA) when it supports the shape, else the window
 * recurrence for Falcon-3 when it does, else the portable CUDA-core chunk
 * path.  GENERIC, TC and SCAN force one (TC and SCAN return
 * FALCON_ERR_UNSUPPORTED for shapes they do not cover).  The tensor-core
 * path covers Falcon-1, 1A, 2 and 2A with bf16 inputs, chunk 64 and
 * d_k = d_v in {64, 128}, Falcon-3A with bf16, chunk 64, d = 64 and
 * 2 <= window <= 16, and Falcon-3 with bf16, chunk 64, d = 64 and
 * 2 <= window <= 9.  SCAN (Falcon-3, 2 <= window <= 8, d_k in {32, 64},
 * d_v a multiple of 16, bf16 or fp32) walks the steps with the state's
 * value columns spread over threads and ignores `chunk`.  TC and SCAN need
 * q, k, v, o and the carried keys / values on 16-byte boundaries: AUTO falls
 * back to the portable path for misaligned tensors, a forced TC or SCAN
 * returns FALCON_ERR_INVALID_ARG. */
typedef enum {
  FALCON_IMPL_AUTO = 0,
  FALCON_IMPL_GENERIC = 1,
  FALCON_IMPL_TC = 2,
  FALCON_IMPL_SCAN = 3
} falcon_impl_t;

enum {
  FALCON_OK = 0,
  FALCON_ERR_INVALID_ARG = -1,   /* null pointer, bad enum, bad size */
  FALCON_ERR_UNSUPPORTED = -2,   /* shape or combination not supported */
  FALCON_ERR_WORKSPACE = -3,     /* workspace missing, too small or misaligned */
  FALCON_ERR_CUDA = -4,          /* a CUDA call or launch failed */
  FALCON_ERR_TIMEOUT = -5        /* a bounded device-side wait expired */
};

typedef struct {
  int32_t B, T, H;      /* batch, tokens in this call, heads (all >= 1; T >= 0 for chunk fwd) */
  int32_t dk, dv;       /* key / value head dims: 16, 32, 64 or 128 */
  int32_t chunk;        /* chunk length of the chunked form: 16, 32 or 64 */
  int32_t window;       /* Falcon-3/3A window W in [1, 64]; ignored otherwise */
  float eps;            /* NLMS regulariser, > 0 (e.g. 1e-6) */
  float eps_gamma;      /* positive-decay floor, in (0, 1] (e.g. 1e-3) */
  int32_t variant;      /* falcon_variant_t */
  int32_t dtype;        /* falcon_dtype_t of q, k, v, o and the carried keys/values */
  int32_t impl;         /* falcon_impl_t (chunk forward only) */
  int32_t pairing;      /* falcon_pairing_t (0 = prefix alignment) */
  int32_t prologue;     /* falcon_prologue_t flags (0 = inputs are features and gates) */
} falcon_params_t;

/* Decode carry: everything the next call needs to continue a sequence.
 * All pointers are device pointers owned by the caller.
 *   S      [B, H, dk, dv] fp32   fast-weight state
 *   k_prev [B, H, dk]     dtype  last key consumed (x of the next pair)
 *   win_x  [B, H, W-1, dk] dtype  window ring of previous pairs' keys  (3/3A, W > 1)
 *   win_v  [B, H, W-1, dv] dtype  window ring of previous pairs' values (3/3A, W > 1)
 *   pos    [B, H]         int64  tokens consumed so far
 * The pair with global index p lives in ring slot p mod (W-1); slots whose
 * pair does not exist (p < 1; with same-step pairing p < 0) hold zeros.  As
 * an input, a NULL carry (or NULL fields) means a fresh sequence: S = 0,
 * k_prev = 0, pos = 0; win_* may be NULL only when no earlier pair exists
 * (pos <= 1, with same-step pairing pos == 0) for every (b, h). */
typedef struct {
  float* S;
  void* k_prev;
  void* win_x;
  void* win_v;
  int64_t* pos;
} falcon_carry_t;

/* Bytes of workspace falcon_chunk_fwd needs for these params (0 if none). */
size_t falcon_workspace_size(const falcon_params_t* p);

/* Chunk-parallel (SSD-style) forward [FW 三种等价形式; JC 三种视角看同一个更新]:
 * the sequence is cut into chunks of `chunk` tokens; inside a chunk the
 * rank-one updates are gathered in the WY representation (Gram matrix of
 * the shifted keys, unit lower-triangular solve), and the state S is carried
 * across chunks with the cumulative log-decay.  Computes o [B, T, H, dv] for
 * the T tokens and, when carry_out is non-NULL, the carry after them
 * (carry_out->S holds the final state S_T; every non-NULL carry_out field
 * is written).  carry_in == NULL starts a fresh sequence.
 * Errors: FALCON_ERR_INVALID_ARG (null q/k/v/beta/lambda/o with T > 0, bad
 * params, carry_in/carry_out overlap), FALCON_ERR_UNSUPPORTED (dims outside
 * {16,32,64,128}, window outside [1,64], forced TC on an unsupported shape),
 * FALCON_ERR_WORKSPACE, FALCON_ERR_CUDA. */
int falcon_chunk_fwd(const falcon_params_t* p, const void* q, const void* k, const void* v,
                     const float* beta, const float* lambda, const falcon_carry_t* carry_in,
                     void* o, falcon_carry_t* carry_out, void* workspace, size_t workspace_bytes,
                     void* stream);

/* falcon_chunk_fwd, plus timing hooks: records the caller's CUDA events
 * (cudaEvent_t handles passed as void*) on `stream`, events[0] before the
 * first kernel of the call and events[i] right after kernel i.  n_events must
 * equal the launch count falcon_chunk_fwd_plan reports plus one.  The work
 * done is exactly that of falcon_chunk_fwd.  Errors: those of
 * falcon_chunk_fwd, and FALCON_ERR_INVALID_ARG for a bad event list. */
int falcon_chunk_fwd_timed(const falcon_params_t* p, const void* q, const void* k, const void* v,
                           const float* beta, const float* lambda, const falcon_carry_t* carry_in,
                           void* o, falcon_carry_t* carry_out, void* workspace,
                           size_t workspace_bytes, void* stream, void* const* events,
                           int32_t n_events);

/* falcon_chunk_fwd for callers that cannot allocate device memory.  The
 * pages have no counterpart to this entry point; it exists for hosts that
 * pass a kernel library only tensors and a stream (plugin interfaces without
 * an allocator, services whose memory budget is fixed once they start
 * serving), which therefore cannot supply falcon_chunk_fwd's workspace.
 *
 * The scratch lives in a fixed 32 MiB array inside the library's device
 * image, held by every device that loads the library until the process
 * exits.  The call itself allocates nothing (no cudaMalloc/cudaFree).
 * Covered: Falcon-1 and Falcon-1A with prologue 0 on the tensor-core path (bf16,
 * d_k = d_v in {64, 128}, chunk 64; see falcon_chunk_fwd_plan) whose
 * falcon_workspace_size is at most 32 MiB: B * H * ceil(T / 64) <= 1927 at
 * d = 64 (17 KB of scratch per chunk) and <= 992 at d = 128 (33 KB per
 * chunk).  Larger problems return FALCON_ERR_WORKSPACE, other variants and
 * shapes FALCON_ERR_UNSUPPORTED (falcon_chunk_fwd serves them; its
 * falcon_workspace_size says whether they need a workspace, 0 for the
 * portable CUDA-core path).  Both are found on the host before anything is
 * enqueued.
 * Every call looks up the array's device address (the first call on a
 * device may also load the library's device code there); make that first
 * call before any stream capture.  All calls share the one array: calls that
 * overlap on the GPU (other streams, other host threads) race and must be
 * serialised by the caller.  The status of the last call is read with
 * falcon_workspace_status(NULL, stream).  Arguments, outputs and other
 * errors as falcon_chunk_fwd. */
int falcon_chunk_fwd_noalloc(const falcon_params_t* p, const void* q, const void* k,
                             const void* v, const float* beta, const float* lambda,
                             const falcon_carry_t* carry_in, void* o, falcon_carry_t* carry_out,
                             void* stream);

/* Bytes of workspace falcon_chunk_fwd_varlen needs for these params
 * (p->B = number of sequences, p->T = their maximum length). */
size_t falcon_varlen_workspace_size(const falcon_params_t* p);

/* Chunk forward over packed sequences of different lengths (varlen), as
 * the chunked framework is used for training [FW 三种等价形式; JC
 * 三种视角看同一个更新].  cu_seqlens (device int32 [B + 1], non-decreasing,
 * cu_seqlens[0] = 0, cu_seqlens[B] = total_tokens) delimits sequence b's
 * tokens [cu_seqlens[b], cu_seqlens[b+1]); every length must be <= p->T.
 * q, k [total_tokens, H, dk], v, o [total_tokens, H, dv], beta
 * [total_tokens, H] (or [total_tokens, H, dv]), lambda [total_tokens, H];
 * carry_in / carry_out are per sequence ([B, H, ...], as for
 * falcon_chunk_fwd; NULL carry_in = every sequence fresh).  On the
 * Falcon-1 / 1A d = 64 tensor-core path (bf16, rows on 16-byte boundaries)
 * the kernels read and write the packed rows in place and take only the
 * chunks that hold tokens (p->prologue applied inside them).  Otherwise the
 * tokens are laid out as a [B, p->T] batch in the workspace (applying
 * p->prologue on the way); positions past a sequence's end get beta = 0 and
 * lambda = 0, steps that neither write nor decay, so each sequence's state
 * after p->T steps is its state after its own length; the same kernel
 * family as falcon_chunk_fwd then runs, and the outputs go back to the
 * packed layout.  carry_out's k_prev, pos and window ring are those after
 * each sequence's own last token.  Errors as falcon_chunk_fwd. */
int falcon_chunk_fwd_varlen(const falcon_params_t* p, const int32_t* cu_seqlens, int64_t total_tokens,
                            const void* q, const void* k, const void* v, const float* beta,
                            const float* lambda, const falcon_carry_t* carry_in, void* o,
                            falcon_carry_t* carry_out, void* workspace, size_t workspace_bytes,
                            void* stream);

/* Which kernel family falcon_chunk_fwd uses for these params
 * (FALCON_IMPL_GENERIC, FALCON_IMPL_TC or FALCON_IMPL_SCAN, written to *impl_out) and how many
 * kernels one call enqueues (*launches_out).  Host-only; either output
 * pointer may be NULL.  Returns FALCON_OK or the error the call would give
 * for these params. */
int falcon_chunk_fwd_plan(const falcon_params_t* p, int32_t* impl_out, int32_t* launches_out);

/* Recurrent form, one token per sequence [FW 三种等价形式 (inference form,
 * O(1) state per step); JC 三种视角看同一个更新]: p->T must be 1.  q, k, v
 * are [B, 1, H, d], beta / lambda [B, 1, H] (or [B, 1, H, dv]).  Updates the
 * carry in place (S, k_prev <- k, window ring push, pos += 1) and writes
 * o [B, 1, H, dv].  carry, carry->S, carry->k_prev and carry->pos are
 * required; win_x / win_v are required for Falcon-3/3A with window > 1.
 * Errors: FALCON_ERR_INVALID_ARG, FALCON_ERR_UNSUPPORTED, FALCON_ERR_CUDA. */
int falcon_recurrent_step(const falcon_params_t* p, const void* q, const void* k, const void* v,
                          const float* beta, const float* lambda, falcon_carry_t* carry, void* o,
                          void* stream);

/* Bytes of workspace falcon_masked_parallel_ref_gpu needs. */
size_t falcon_masked_parallel_workspace_size(const falcon_params_t* p);

/* Masked-parallel form of a fresh sequence [FW 三种等价形式 (linear attention
 * (phi(Q) phi(K)^T (.) M) V without denominator); JC 三种视角看同一个更新]:
 * the whole T x T decay mask from the global cumulative log-decay and, for
 * the regression variants, one unit lower-triangular solve over all T
 * steps (T*W unknowns for Falcon-3).  fp32 arithmetic, quadratic cost: a
 * reference for tests, limited to T <= 1024 (T*window <= 2048).  Writes
 * o [B, T, H, dv] and S_final [B, H, dk, dv] (fp32).
 * Errors: FALCON_ERR_INVALID_ARG, FALCON_ERR_UNSUPPORTED (T too large),
 * FALCON_ERR_WORKSPACE, FALCON_ERR_CUDA. */
int falcon_masked_parallel_ref_gpu(const falcon_params_t* p, const void* q, const void* k,
                                   const void* v, const float* beta, const float* lambda, void* o,
                                   float* S_final, void* workspace, size_t workspace_bytes,
                                   void* stream);

/* Bytes of workspace falcon_backward needs for these params (0 when the
 * params are invalid or not covered). */
size_t falcon_backward_workspace_size(const falcon_params_t* p);

/* Gradient of the chunk forward, for training in the chunked framework
 * [FW 三种等价形式; JC 三种视角看同一个更新] (the pages give the forward
 * only; the backward is the chain rule through the update written at the
 * top of this header, Falcon-3/3A's window of pairs included).  For the loss
 * L = <o, dO> + <S_T, dS_final> of falcon_chunk_fwd(p, q, k, v, beta,
 * lambda, carry_in) it writes
 *   dq, dk [B, T, H, dk], dv [B, T, H, dv] (the params' dtype),
 *   dbeta (the shape of beta), dlambda [B, T, H] (fp32),
 * and, through the fields of dcarry (NULL, or any field NULL, skips them):
 *   dcarry->S      [B, H, dk, dv] fp32  gradient of carry_in->S,
 *   dcarry->k_prev [B, H, dk] dtype      gradient of carry_in->k_prev,
 *   dcarry->win_x  [B, H, W-1, dk], dcarry->win_v [B, H, W-1, dv] dtype
 *                  gradients of the carried window ring (Falcon-3/3A, W > 1;
 *                  both or neither; slot layout as in the carry);
 * dcarry->pos is ignored.  dO has the shape and dtype of o; dS_final (fp32
 * [B, H, dk, dv]) may be NULL (zero).  carry_in supplies S, k_prev, the
 * window ring and pos as for the forward (NULL = fresh sequence); a key or
 * ring entry that no existing pair reads gets a zero gradient.  The decay
 * clamp passes the gradient where eps_gamma <= 1 - lambda <= 1.  The forward
 * is recomputed inside (states kept at every 64th step in the workspace), so
 * o need not be saved.  Covered: every variant, both pairings, bf16 or fp32,
 * d_k = d_v in {32, 64, 128}; Falcon-3/3A with W up to 64 (up to 34 at
 * d = 128, the window kernel's shared memory); any T >= 0 (chunk and impl
 * are ignored).  Falcon-1/1A at d = 64 run a chunked kernel, Falcon-3/3A
 * and d = 128 a step-by-step kernel that carries the window's key and value
 * gradients in a ring, the rest a step-by-step one-pair kernel.  Gradients
 * must not overlap inputs or one another.  The chunked kernel with bf16
 * inputs runs its products on the tensor cores with bounded waits: a wait
 * that runs out is recorded in the workspace's status word and read with
 * falcon_workspace_status, as for the chunk forward.
 * Errors: FALCON_ERR_INVALID_ARG, FALCON_ERR_UNSUPPORTED (other dims, the
 * prologue, a window past the limit), FALCON_ERR_WORKSPACE, FALCON_ERR_CUDA. */
int falcon_backward_carry(const falcon_params_t* p, const void* q, const void* k, const void* v,
                          const float* beta, const float* lambda, const falcon_carry_t* carry_in,
                          const void* dO, const float* dS_final, void* dq, void* dk, void* dv,
                          float* dbeta, float* dlambda, const falcon_carry_t* dcarry, void* workspace,
                          size_t workspace_bytes, void* stream);

/* falcon_backward_carry with dcarry = {dS_in, dk_prev} (no ring gradients):
 * dS_in [B, H, dk, dv] fp32 and dk_prev [B, H, dk] dtype may each be NULL. */
int falcon_backward(const falcon_params_t* p, const void* q, const void* k, const void* v,
                    const float* beta, const float* lambda, const falcon_carry_t* carry_in,
                    const void* dO, const float* dS_final, void* dq, void* dk, void* dv,
                    float* dbeta, float* dlambda, float* dS_in, void* dk_prev, void* workspace,
                    size_t workspace_bytes, void* stream);

/* Status of the last tensor-core chunk forward that used `workspace`
 * (falcon_chunk_fwd_plan reports FALCON_IMPL_TC for it; falcon_chunk_fwd,
 * _timed, _varlen), or, with workspace == NULL, of the last
 * falcon_chunk_fwd_noalloc call on the current device.  The pages have no
 * counterpart: this is the library's failure detection.  Every wait of
 * those kernels on another warp, a copy or a product is bounded in time
 * (2 s); a wait that runs out makes its kernel record a timeout in the
 * status word (the first 4 bytes of the workspace), skip its remaining
 * chunks, wait for its own copies in flight, free its tensor memory and
 * return, and the kernels after it in the call compute nothing.  The call
 * itself returned FALCON_OK before the kernels ran, so this is how the
 * caller learns of it.  Each such call clears the word when it starts.
 * The function synchronises `stream` (the call's stream), reads the word
 * and clears it.  Returns FALCON_OK, FALCON_ERR_TIMEOUT (the outputs and
 * carry of that call are incomplete), FALCON_ERR_WORKSPACE (workspace not
 * 256-byte aligned) or FALCON_ERR_CUDA.  The chunked backward (Falcon-1 /
 * 1A, d = 64) keeps its word in the same place.  Other kernel families have
 * no device-side waits and do not write the word. */
int falcon_workspace_status(const void* workspace, void* stream);

/* Test hook of the failure-detection path (no counterpart on the pages; not
 * for production use).  wait_limit_ns > 0 sets the limit of the bounded
 * device-side waits of the Falcon-1 / 1A, 3 and 3A tensor-core kernels
 * and of the chunked backward launched from now on in this process (0
 * restores 2 s; the Falcon-2 kernel keeps 2 s).  stall != 0 makes the next
 * forward call's per-chunk kernel wait once, before it loads anything, on a barrier
 * that nothing completes: that wait runs out after the limit, the timeout is
 * recorded as described at falcon_workspace_status and the call's later
 * kernels skip their work.  No fault, trap or unbounded wait is involved;
 * the CUDA context stays usable.  Process-wide; not thread-safe against
 * concurrent calls that should not see it. */
void falcon_test_hooks(uint64_t wait_limit_ns, int32_t stall);

/* Static description of an error code (never NULL). */
const char* falcon_strerror(int code);

/* Library version string, e.g. "falcon-gb300 0.1 sm_103a". */
const char* falcon_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FALCON_H */
