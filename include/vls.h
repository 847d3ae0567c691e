/*
 * vls.h -- C ABI of libvls, row-wise vocabulary log-softmax statistics on
 * NVIDIA GB300 (sm_103a).
 *
 * A "row" is one token's logits over the vocabulary: N rows of V contiguous
 * columns.  Where each row starts is given by a vls_rows descriptor (below):
 * one row stride, or two strides for a [B, T, V] tensor read as N = B*T rows,
 * so that slices such as logits[:, :V] or logits[:, :-1, :] are read in place.
 * Every call computes in fp32 with one rounding at each store.  The softmax
 * statistics are taken in one read of the logits (online max and sum of
 * exponentials, "Add Triton kernels for vocab-parallel logprobs, entropy and
 * KL", DeepSpeed PR #8838, section Changes and review "Suggested change");
 * each forward saves per-row (max, log-sum-exp) so that its backward is one
 * read of the logits plus one write of the gradient.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Pointers: all data pointers are DEVICE pointers (cudaMalloc'd, or
 *    managed memory) on one device.  The caller owns every buffer; the
 *    library allocates, frees and synchronises nothing.
 *  - Stream: `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *    default stream).  Every call only enqueues work on it and returns.
 *  - Device guard: the launch goes to the device that holds the first input
 *    pointer, whatever device is current; the current device is restored
 *    before returning ("perf(logp): fused zero-workspace backward ...",
 *    RL-Kernel PR #495, review "Hardening Proposals").  The stream must
 *    belong to that device.
 *  - Inputs are never written.  Outputs must not overlap inputs.
 *  - N == 0 (or n == 0) returns VLS_OK without touching any pointer and
 *    without a launch.
 *  - Logits are finite or -inf (a mask).  A row whose logits are all -inf
 *    has no distribution: its statistics and gradient row are NaN.  A NaN
 *    logit makes every statistic and gradient of its row NaN.
 *  - cap: 0 means no softcap.  cap > 0 applies y = cap*tanh(x/cap) to every
 *    logit before the softmax, in registers ("Final Logit Softcap",
 *    section Summary); -inf logits then become -cap.  A capped logit
 *    carries an absolute error of a few 1e-7 * cap, so the results keep
 *    the fp32 accuracy rule at caps of the usual size (tested from 4 to 100).
 *  - Results are deterministic and batch invariant: a row's outputs depend
 *    only on that row's data, V and the dtype, bit for bit, not on N, on the
 *    row's position or on the alignment of the row in memory.
 *  - CUDA graphs: the calls may be recorded by stream capture (any capture
 *    mode).  While `stream` is capturing, the launch goes to the current
 *    device and pointers are not checked against it (the runtime refuses
 *    those queries inside a capture).  Make one call of each kind before
 *    capturing, so the first-use set-up of the tensor-core kernels happens
 *    outside it.
 *  - Errors: each call returns VLS_OK (0) or one of the VLS_ERR_* codes
 *    below; it never aborts, throws or prints.  Argument errors are found
 *    before any CUDA call.  vls_status_string() names a code.
 */
#ifndef VLS_H_
#define VLS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of logits, gradients and softcap tensors. */
typedef enum { VLS_F32 = 0, VLS_BF16 = 1, VLS_F16 = 2 } vls_dtype;

/* VLS_KL_REVERSE: KL(p_a || p_b); VLS_KL_FORWARD: KL(p_b || p_a).  In both the
 * gradient flows to `a` (the policy) only; `b` (the reference) is detached
 * (DeepSpeed PR #8838, review by @0z5a: "reverse KL with a detached
 * teacher"). */
typedef enum { VLS_KL_REVERSE = 0, VLS_KL_FORWARD = 1 } vls_kl_dir;

/* Per-row statistics a forward saves for its backward: m = max_j z_j and
 * log_s = log(sum_j exp(z_j - m)), so log p_j = (z_j - m) - log_s.  Kept as
 * the pair rather than m + log_s so that the backward's (z - m) - log_s never
 * adds a large common offset into an fp32 sum.  8 bytes per row. */
typedef struct { float m; float log_s; } vls_rowstat;

/* Row addressing of a logits operand: row r (0 <= r < N) starts
 *     (r / group) * ld_group + (r % group) * ld
 * elements after the operand's base pointer, and its V columns are
 * contiguous.  A plain [N, V] matrix with row stride ld is {ld, 0, 0} (group
 * 0: all rows form one group).  A [B, T, V] tensor with element strides
 * (sB, sT, 1), read as N = B*T rows, is {sT, T, sB}: a slice such as
 * x[:, :-1, :] keeps its two strides and is read in place where a single row
 * stride would need a copy ("Add Triton kernels for vocab-parallel logprobs,
 * entropy and KL", DeepSpeed PR #8838, review "Suggested change": rows
 * addressed with up to two strides).  Requires ld >= V, group >= 0 and, when
 * group > 0, ld_group >= V.  Rows may overlap: operands are only read.
 * Gradients are always written as [N, V] contiguous. */
typedef struct { int64_t ld; int64_t group; int64_t ld_group; } vls_rows;

enum {
  VLS_OK = 0,
  VLS_ERR_NULL = 1,     /* a required pointer (or vls_rows) is NULL (with N > 0) */
  VLS_ERR_SHAPE = 2,    /* N < 0, V < 1, a vls_rows field out of range, k < 1 or
                           k > VLS_MAX_TOPK, n < 0,
                           R < 1, a shard outside [0, V_total)                   */
  VLS_ERR_DTYPE = 3,    /* dtype not a vls_dtype; gy dtype neither F32 nor dt     */
  VLS_ERR_CAP = 4,      /* cap NaN, infinite or negative (softcap calls: cap <= 0) */
  VLS_ERR_DEVICE = 5,   /* a pointer is not device memory, or pointers / stream
                           sit on different devices                               */
  VLS_ERR_LAUNCH = 6,   /* the CUDA launch failed (cudaGetLastError after launch) */
  VLS_ERR_ARG = 7,      /* another bad argument (e.g. an unknown KL direction)    */
  VLS_ERR_TOO_LARGE = 8, /* the call needs more than the fixed scratch of
                           vls_linear_logp_fwd_noalloc                            */
  VLS_ERR_TIMEOUT = 9   /* vls_check_device_error: a bounded wait in a tensor-core
                           kernel ran out (its outputs are invalid)               */
};

/* Largest top-k the logprob calls accept. */
#define VLS_MAX_TOPK 1024

/* ------------------------------------------------------------------------ */
/* Final-logit softcap, standalone ("Final Logit Softcap", Summary and       */
/* Tensor and Precision Contract).                                           */
/* ------------------------------------------------------------------------ */

/* y[i] = cap * tanh(x[i] / cap) for i in [0, n); x and y are n contiguous
 * elements of dtype dt (y may not alias x).  fp32 math, one cast at the
 * store.  cap must be finite and > 0 (the page's constructor check). */
int vls_softcap_fwd(const void* x, void* y, int64_t n, vls_dtype dt, float cap, void* stream);

/* gx[i] = gy[i] * (1 - tanh^2(x[i] / cap)); the cap cancels in the derivative
 * ("Final Logit Softcap", Summary).  x and gx have dtype dt; gy has dtype
 * gy_dt, which is VLS_F32 or dt.  tanh is recomputed from the saved input. */
int vls_softcap_bwd(const void* x, const void* gy, vls_dtype gy_dt, void* gx, int64_t n,
                    vls_dtype dt, float cap, void* stream);

/* ------------------------------------------------------------------------ */
/* Target log-probabilities (DeepSpeed PR #8838, Changes; RL-Kernel PR #495, */
/* Summary and Behavior changes).                                            */
/* ------------------------------------------------------------------------ */

/* logp[r*k + j] = log_softmax(z_r)[ids[r*k + j]] (fp32) for each of the k ids
 * of row r, where z_r is row r of `logits` (after the softcap when cap > 0).
 * An id is ignored when it equals ignore_index or lies outside [0, V); its
 * logp is exactly 0.  ids: int64 [N, k] contiguous.  stats: [N], written for
 * the backward.  1 <= k <= VLS_MAX_TOPK. */
int vls_logp_fwd(const void* logits, const vls_rows* rows, vls_dtype dt, int64_t N, int64_t V,
                 const int64_t* ids, int32_t k, int64_t ignore_index, float cap,
                 float* logp, vls_rowstat* stats, void* stream);

/* Vector-Jacobian product of vls_logp_fwd for upstream g (fp32 [N, k]):
 *   dlogits[r, c] = (sum over valid j with ids[r, j] == c of g[r, j]
 *                    - G_r * p_r[c]) * dz/dx,
 *   G_r = sum over valid j of g[r, j],  p_r = softmax(z_r),
 * the one-hot terms of duplicate ids added in ascending j in fp32 before the
 * single cast (DeepSpeed PR #8838, Changes).  A row without a valid id is
 * written as exact zeros (RL-Kernel PR #495, Behavior changes).  dlogits:
 * [N, V] contiguous, dtype dt.  stats: as written by vls_logp_fwd with the
 * same logits, cap and dtype. */
int vls_logp_bwd(const void* logits, const vls_rows* rows, vls_dtype dt, int64_t N, int64_t V,
                 const int64_t* ids, int32_t k, int64_t ignore_index, float cap,
                 const float* g, const vls_rowstat* stats, void* dlogits, void* stream);

/* ------------------------------------------------------------------------ */
/* Entropy (DeepSpeed PR #8838, review "Suggested change": H = log S - W/S). */
/* ------------------------------------------------------------------------ */

/* H[r] = -sum_c p_r[c] log p_r[c] (fp32 [N]); stats [N] for the backward. */
int vls_entropy_fwd(const void* logits, const vls_rows* rows, vls_dtype dt, int64_t N, int64_t V,
                    float cap, float* H, vls_rowstat* stats, void* stream);

/* dlogits[r, c] = -g[r] * p_r[c] * (log p_r[c] + H[r]) * dz/dx, 0 on -inf
 * columns.  g, H: fp32 [N]; dlogits: [N, V] contiguous, dtype dt. */
int vls_entropy_bwd(const void* logits, const vls_rows* rows, vls_dtype dt, int64_t N, int64_t V,
                    float cap, const float* g, const float* H, const vls_rowstat* stats,
                    void* dlogits, void* stream);

/* ------------------------------------------------------------------------ */
/* KL divergence (DeepSpeed PR #8838, review "Suggested change":             */
/* KL = W/S_A - log S_A + log S_B).                                          */
/* ------------------------------------------------------------------------ */

/* kl[r] (fp32 [N]) between softmax(a_r) and softmax(b_r), in direction dir.
 * +inf when the first distribution supports a column that the second masks
 * (-inf logit), decided on the logits; NaN when a row of a or b is all -inf.
 * a and b: same dtype, each addressed by its own vls_rows.  stats_a, stats_b:
 * [N] for the backward. */
int vls_kl_fwd(const void* a, const vls_rows* rows_a, const void* b, const vls_rows* rows_b, vls_dtype dt,
               int64_t N, int64_t V, vls_kl_dir dir, float cap, float* kl,
               vls_rowstat* stats_a, vls_rowstat* stats_b, void* stream);

/* Gradient of g[r] * kl[r] with respect to a:
 *   reverse: da[r, c] = g p_a[c] ((log p_a[c] - log p_b[c]) - kl[r]) * dz/dx,
 *            0 where a = -inf, a NaN row when kl[r] is +inf or NaN;
 *   forward: da[r, c] = g (p_a[c] - p_b[c]) * dz/dx, a NaN row when kl[r] is NaN.
 * g, kl: fp32 [N]; da: [N, V] contiguous, dtype dt. */
int vls_kl_bwd(const void* a, const vls_rows* rows_a, const void* b, const vls_rows* rows_b, vls_dtype dt,
               int64_t N, int64_t V, vls_kl_dir dir, float cap, const float* g,
               const float* kl, const vls_rowstat* stats_a, const vls_rowstat* stats_b,
               void* da, void* stream);

/* ------------------------------------------------------------------------ */
/* Fused statistics: target logprobs, entropy and KL of the same policy      */
/* logits from one read of the policy (and one of the reference), and one    */
/* backward pass for any weighted sum of them.  The quantities are the ones  */
/* above; RL and distillation losses take them together (DeepSpeed PR #8838, */
/* Changes: logprobs, entropy and KL over the same shard).                   */
/* ------------------------------------------------------------------------ */

/* Forward.  a: policy logits; b: reference logits (NULL when kl is NULL).
 * logp [N, k] (NULL to skip; needs ids), H [N] (NULL to skip), kl [N] in
 * direction dir (NULL to skip).  stats_a [N] always; stats_b [N] with kl.
 * Each output equals the corresponding single call's. */
int vls_fused_fwd(const void* a, const vls_rows* rows_a, const void* b, const vls_rows* rows_b,
                  vls_dtype dt, int64_t N, int64_t V,
                  const int64_t* ids, int32_t k, int64_t ignore_index, vls_kl_dir dir, float cap,
                  float* logp, float* H, float* kl, vls_rowstat* stats_a, vls_rowstat* stats_b,
                  void* stream);

/* Backward: da = d/da of sum_r [ sum_j g_logp[r,j] logp[r,j] + g_H[r] H[r]
 * + g_kl[r] KL[r] ], the sum of the single calls' gradients computed in fp32
 * and cast once.  A term is left out when its upstream pointer is NULL
 * (g_logp needs ids; g_H needs H; g_kl needs b, kl and stats_b).  da: [N, V]
 * contiguous, dtype dt. */
int vls_fused_bwd(const void* a, const vls_rows* rows_a, const void* b, const vls_rows* rows_b,
                  vls_dtype dt, int64_t N, int64_t V,
                  const int64_t* ids, int32_t k, int64_t ignore_index, vls_kl_dir dir, float cap,
                  const float* g_logp, const float* g_H, const float* g_kl, const float* H, const float* kl,
                  const vls_rowstat* stats_a, const vls_rowstat* stats_b, void* da, void* stream);

/* ------------------------------------------------------------------------ */
/* Vocabulary-parallel statistics, split phase (DeepSpeed PR #8838, Changes: */
/* local max and sum-exp from one read, rescaled to the global max, so that  */
/* tensor parallelism needs one MAX and one SUM all-reduce; review           */
/* "Suggested change": entropy / KL sums re-centred on the global max, the   */
/* support-mismatch flag sharing the MAX all-reduce).                        */
/*                                                                           */
/* Each rank holds the columns [vocab_offset, vocab_offset + V_shard) of a   */
/* V_total-column vocabulary.  vls_*_partial sweeps its shard once and       */
/* writes one vls_partial per row; the caller gathers the R ranks' partial   */
/* arrays in rank order into one [R, N] array (an all-gather of 24 bytes per */
/* row per rank) and vls_*_combine folds them in rank order 0..R-1 and       */
/* writes the same outputs and per-row statistics as the unsharded forward.  */
/* The backward then runs per shard: vls_entropy_bwd / vls_kl_bwd unchanged  */
/* on the shard with the combined statistics, vls_logp_bwd_shard for logp.   */
/* V_shard = 0 (an empty shard) is allowed and gives the identity partial;   */
/* its logits pointer and vls_rows may then be NULL.                         */
/* Results are deterministic for a fixed sharding; they match the unsharded  */
/* call up to rounding (the reduction tree differs).                         */
/* ------------------------------------------------------------------------ */

/* Per-row partial state of one shard, centred on the shard's maxima.
 * logp: m, s.  entropy: m, s, w = sum e^{z-m}(z-m).  KL(P||Q) (P the first
 * argument of the direction): m, s of P, w = sum e^{p-m}((p-m)-(q-mq)),
 * mq, sq of Q, flag = a column with P finite and Q = -inf. */
typedef struct {
  float m, s, w, mq, sq;
  uint32_t flag;
} vls_partial;

/* Partial of vls_logp_fwd over a shard.  part: [N].  zt: fp32 [N, k]; for an
 * id that is valid against V_total and lies in this shard, the raw (uncapped)
 * logit of that column, else 0 -- summed over the ranks it is the target's
 * logit (exactly one rank owns a valid id). */
int vls_logp_partial(const void* logits, const vls_rows* rows, vls_dtype dt, int64_t N, int64_t V_shard,
                     int64_t vocab_offset, int64_t V_total, const int64_t* ids, int32_t k,
                     int64_t ignore_index, float cap, vls_partial* part, float* zt, void* stream);

/* Folds parts [R, N] (rank-major) and zt [R, N, k] into logp [N, k] and stats [N]. */
int vls_logp_combine(const vls_partial* parts, const float* zt, int32_t R, int64_t N, const int64_t* ids,
                     int32_t k, int64_t V_total, int64_t ignore_index, float cap, float* logp,
                     vls_rowstat* stats, void* stream);

/* vls_logp_bwd for a shard: ids are global column indices (valid against
 * V_total); the one-hot terms land in this shard's columns only, while G
 * sums the upstream gradients of every valid id.  dlogits: [N, V_shard]
 * contiguous.  stats: from vls_logp_combine. */
int vls_logp_bwd_shard(const void* logits, const vls_rows* rows, vls_dtype dt, int64_t N, int64_t V_shard,
                       int64_t vocab_offset, int64_t V_total, const int64_t* ids, int32_t k,
                       int64_t ignore_index, float cap, const float* g, const vls_rowstat* stats,
                       void* dlogits, void* stream);

int vls_entropy_partial(const void* logits, const vls_rows* rows, vls_dtype dt, int64_t N, int64_t V_shard,
                        float cap, vls_partial* part, void* stream);

/* Folds parts [R, N] into H [N] and stats [N]. */
int vls_entropy_combine(const vls_partial* parts, int32_t R, int64_t N, float* H, vls_rowstat* stats,
                        void* stream);

int vls_kl_partial(const void* a, const vls_rows* rows_a, const void* b, const vls_rows* rows_b,
                   vls_dtype dt, int64_t N, int64_t V_shard, vls_kl_dir dir, float cap, vls_partial* part, void* stream);

/* Folds parts [R, N] into kl [N], stats_a [N], stats_b [N] (dir as in the partials). */
int vls_kl_combine(const vls_partial* parts, int32_t R, int64_t N, vls_kl_dir dir, float* kl,
                   vls_rowstat* stats_a, vls_rowstat* stats_b, void* stream);

/* ------------------------------------------------------------------------ */
/* Fused linear head + target log-probabilities.  The pages name a           */
/* linear_logp op without defining it ("perf(logp): fused zero-workspace     */
/* backward ...", RL-Kernel PR #495, Summary); it is read here as the        */
/* logprobs of the logits z = h @ W^T of a linear vocabulary head, where z   */
/* is never written to memory.  The tensor cores (tcgen05) form z tile by    */
/* tile and the statistics of vls_logp_fwd are folded from those tiles.      */
/* The forward is split phase: the vocabulary is cut into fixed chunks       */
/* (vls_linear_logp_chunks), vls_linear_logp_partial writes one vls_partial  */
/* per chunk and row plus the owned targets' logits, and vls_logp_combine    */
/* (R = the chunk count, V_total = V) folds them in chunk order into logp    */
/* and stats, exactly as for vocabulary shards.                              */
/* ------------------------------------------------------------------------ */

/* Largest top-k the linear call accepts. */
#define VLS_LINEAR_MAX_TOPK 16

/* Number of vocabulary chunks S of a V-column head (a function of V only, so
 * results do not depend on N); parts and zt of vls_linear_logp_partial hold
 * S rows of N entries.  Returns -1 when V < 1. */
int64_t vls_linear_logp_chunks(int64_t V);

/* h: [N, D] hidden states, row stride ldh; W: [V, D] head weights, row
 * stride ldw; both of dtype dt, VLS_BF16 or VLS_F16 (fp32 accumulation).
 * h, W and their row strides must be 16-byte aligned (ldh, ldw multiples of
 * 8 elements), as the tensor-memory-access loads require.  ids: int64 [N, k],
 * 1 <= k <= VLS_LINEAR_MAX_TOPK, ignored as in vls_logp_fwd.  part: [S, N];
 * zt: fp32 [S, N, k] (the raw logit of each valid id in the chunk that holds
 * it, 0 in the others).  status: one device uint32 the caller zeroes; the
 * kernel sets bit 0 if one of its internal waits ran out (a fault of the
 * kernel, not of the inputs), and the partials are then invalid.  Needs a
 * GPU with tcgen05 (sm_100 family); the library is built for sm_103a. */
int vls_linear_logp_partial(const void* h, int64_t ldh, const void* W, int64_t ldw, vls_dtype dt,
                            int64_t N, int64_t D, int64_t V, const int64_t* ids, int32_t k,
                            int64_t ignore_index, vls_partial* part, float* zt, uint32_t* status,
                            void* stream);

/* Bytes of device workspace vls_linear_logp_bwd needs: dz [N, V] in the
 * operand dtype, its rows padded to a multiple of 8 elements, rounded up to
 * 256 bytes (about 2 N V).  Returns -1 for sizes out of range. */
int64_t vls_linear_logp_bwd_workspace(int64_t N, int64_t D, int64_t V);

/* Gradients of sum_{r,j} g[r, j] logp[r, j] with respect to h and W, where
 * logp is vls_linear_logp's output for the same h, W, ids and ignore_index
 * and stats its (m, log S):
 *     dz = g one-hot - G p   (G = sum of the valid g of the row),
 *     dh = dz @ W  [N, D],   dW = dz^T @ h  [V, D],
 * with the logits recomputed on the tensor cores from h and W.  dz is formed
 * in fp32 and rounded once to dt before the two products, which accumulate
 * in fp32 and round once to dt at the store.  g: fp32 [N, k]; dh, dW:
 * contiguous, dtype dt, overlapping neither each other, the inputs nor the
 * workspace (rows that are 16-byte multiples on 16-byte aligned bases are
 * stored through TMA, others by the threads).  workspace: at least
 * vls_linear_logp_bwd_workspace(N, D, V) bytes, 256-byte aligned, the
 * caller's; its contents on entry do not matter.  When the rows are too few
 * to fill the GPU, dh is summed in K runs (split-K) whose fp32 partial sums
 * are kept in dW's memory before dW is computed; dh's rounding then depends
 * on N and on the GPU's SM count, within the same fp32 bound.  status as for
 * vls_linear_logp_partial.  N, D and V are at most 2^31 - 512. */
int vls_linear_logp_bwd(const void* h, int64_t ldh, const void* W, int64_t ldw, vls_dtype dt, int64_t N,
                        int64_t D, int64_t V, const int64_t* ids, int32_t k, int64_t ignore_index,
                        const float* g, const vls_rowstat* stats, void* dh, void* dW, void* workspace,
                        int64_t workspace_bytes, uint32_t* status, void* stream);

/* The whole linear-head logprob forward (the partial call, then the combine)
 * without any buffer from the caller beyond its inputs and outputs.  The
 * pages have no counterpart to this call: it exists for callers that cannot
 * allocate device memory, such as a serving engine that has given all of it
 * to its own pool and forbids further cudaMalloc calls, or a program held to
 * a fixed device-memory budget.  The intermediate partials live in one fixed
 * array of the library (32 MiB), which bounds a call: N * S <= 2^20 and
 * N * S * k <= 2^21 with S = vls_linear_logp_chunks(V) (for V = 151936,
 * S = 75: up to 13981 rows at k = 1); larger calls return VLS_ERR_TOO_LARGE
 * before touching the GPU.  Arguments, outputs and status are those of
 * vls_linear_logp_partial and vls_logp_combine: logp [N, k] and stats [N].
 * The array is held until the process exits on every GPU where it is
 * loaded: with CUDA's lazy module loading (the default) each GPU where this
 * call has been made, with eager loading (CUDA_MODULE_LOADING=EAGER) every
 * GPU the process uses, from the moment the library loads.  It is the
 * library's own memory, not counted as the call's peak extra memory.
 * The first call on a device looks up the array's address there (a runtime
 * query, no allocation), so make that first call before any stream capture.
 * The launch device is chosen as for the other calls.  Every call uses the
 * same array: calls whose work overlaps on the GPU (on different streams or
 * from different threads) race and must be ordered by the caller. */
int vls_linear_logp_fwd_noalloc(const void* h, int64_t ldh, const void* W, int64_t ldw, vls_dtype dt,
                                int64_t N, int64_t D, int64_t V, const int64_t* ids, int32_t k,
                                int64_t ignore_index, float* logp, vls_rowstat* stats, uint32_t* status,
                                void* stream);

/* ------------------------------------------------------------------------ */
/* Status                                                                    */
/* ------------------------------------------------------------------------ */

/* Static, NUL-terminated name of a status code ("VLS_OK", ...); never NULL. */
const char* vls_status_string(int status);

/* Reports failures of work already enqueued on the CURRENT device, which the
 * calls themselves cannot return because they only enqueue it.  Synchronises
 * the device (cudaDeviceSynchronize), then reads the library's status word
 * on it.  Every wait of the tensor-core kernels (the vls_linear_logp_* calls)
 * is bounded in time; one that runs out makes the kernel drain the copies
 * and products it has in flight and return early, and sets bit 0 both of
 * the call's own status word and of this library word.  A failed kernel is
 * reported, never replaced by another path ("Final Logit Softcap", section
 * Backends: a failed launch is not retried with another backend, fallback
 * happens only when a backend cannot be loaded).  Returns VLS_ERR_TIMEOUT
 * when that happened since the last call that returned it (the word is then
 * cleared),
 * VLS_ERR_LAUNCH when the synchronisation reports a CUDA error of earlier
 * work, else VLS_OK.  It synchronises, so it must not be called while a
 * stream of the device is being captured into a graph; call it when no
 * tensor-core call is in flight from another thread (a bit set between the
 * read and the clear would be lost).  The row kernels have no waits of
 * their own: their only cross-CTA synchronisation is the hardware cluster
 * barrier, which every CTA of a cluster reaches. */
int vls_check_device_error(void);

/* Library version, major*10000 + minor*100 + patch. */
int vls_version(void);

#ifdef __cplusplus
}
#endif

#endif /* VLS_H_ */
