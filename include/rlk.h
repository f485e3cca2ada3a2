/*
 * rlk.h -- C ABI of the GB300 (sm_103a) fused linear selected-token log-prob.
 *
 * What it computes.  For hidden states h[N,H] and LM-head weights W[V,H]
 * (both bf16), target ids y[N], an active mask and a rollout temperature T:
 *
 *     s[t,v]  = sum_k h[t,k] * W[v,k]                 (fp32 accumulation)
 *     logp[t] = s[t,y_t]/T - log( sum_v exp(s[t,v]/T) )   for active t
 *
 * without ever storing the [N,V] logits ("RL-Kernel Roadmap (2026)", P0.2
 * "Typical Fused Operators": fused CE log-prob that never lands [B,S,V]
 * logits, forward streaming vocab blocks with an online softmax, backward
 * recomputing tiles), with the explicit max / sum-exp / target-logit merge
 * and full-gradient backward of "RL-Kernel integration roadmap for vime",
 * Operator Integration Plan, "linear_logp / lm_head + logp", and the masked
 * dlogp diagnostics of the same page's "Consistency Contract".
 *
 * Conventions shared by every entry point.
 *  - Ownership: every array argument is a caller-owned DEVICE pointer unless
 *    stated otherwise.  The library never allocates, frees or synchronises;
 *    scratch memory is the caller's `workspace`, sized by the matching
 *    *_workspace_bytes() query.  Work is enqueued on `stream` and is visible
 *    once the caller synchronises that stream.
 *  - Layout: contiguous row-major.  bf16 matrices (hidden, weight, dhidden,
 *    dweight) must start on a 16-byte boundary; workspace on 256 bytes.
 *  - Mask bytes: nonzero = active.  A NULL mask means every row is active.
 *    Targets of inactive rows are never read.
 *  - Shapes: H must be a positive multiple of 64; 1 <= V <= 2^31 - 2^16;
 *    0 <= N <= 2^31 - 2^16 (device indices are 32-bit, with headroom for
 *    rounding N and V up to whole tiles).  N = 0 returns RLK_OK without
 *    launching anything.
 *  - Errors: argument errors are returned synchronously, before anything is
 *    enqueued; a failed launch returns RLK_ERR_LAUNCH.  There is no fallback
 *    path: an unsupported case is an error, never a silent slower route.
 *    Data errors found on the device (an active row whose target lies
 *    outside [0, V)) set bits in *device_error_word (if not NULL; the caller
 *    zeroes it) and give that row logp = NaN.
 *  - Determinism: tile shapes, vocab-chunk widths and every reduction order
 *    are compile-time constants, never functions of N, the mask or the SM
 *    count, and no floating-point atomics are used.  A row's logp, lse and
 *    dhidden are therefore bitwise identical whatever batch it is scored in;
 *    dweight is bitwise reproducible for identical inputs.
 */
#ifndef RLK_H_
#define RLK_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RLK_OK = 0,
    RLK_ERR_INVALID_VALUE = 1,   /* NULL / misaligned pointer, bad size, T not finite > 0 */
    RLK_ERR_UNSUPPORTED = 2,     /* H % 64 != 0, too large, or the device is not sm_103 */
    RLK_ERR_WORKSPACE = 3,       /* workspace NULL, misaligned or smaller than the query */
    RLK_ERR_LAUNCH = 4,          /* a CUDA launch or attribute call failed */
} rlk_status_t;

/* bits of *device_error_word */
#define RLK_DEVERR_TARGET_RANGE 0x1u   /* an active row's target id is outside [0, V) */
#define RLK_DEVERR_WAIT_TIMEOUT 0x2u   /* a pipeline wait gave up (the results are invalid) */
#define RLK_DEVERR_ROW_RANGE 0x4u      /* an entry of a row-index list is outside [0, N) */

/* element type of rlk_logp_from_logits' logits */
#define RLK_DTYPE_F32 0
#define RLK_DTYPE_BF16 1

/* Result of rlk_dlogp_audit, written to device memory. */
typedef struct {
    int64_t active_count;   /* number of active tokens (exact) */
    int64_t argmax_index;   /* lowest token index attaining max |d|; -1 if none is active */
    double mean_dlogp;      /* sum d / count   (NaN when count == 0) */
    double approx_kl;       /* sum (exp(d) - 1 - d) / count   (NaN when count == 0) */
    float max_abs_dlogp;    /* max |d| over active tokens (0 when none; NaN ranks highest) */
    uint32_t error_flags;   /* bit 0: an active d was not finite */
} rlk_audit_result_t;

/* Result of rlk_grpo_clip_loss, written to device memory. */
typedef struct {
    int64_t active_count;   /* number of active tokens */
    int64_t clipped_count;  /* active tokens where the clipped term is selected (zero gradient) */
    int64_t outside_count;  /* active tokens with r outside [1 - eps_low, 1 + eps_high] */
    double loss;            /* -loss_scale * sum_active min(r A, clip(r) A) */
    double mean_ratio;      /* sum_active r / active_count   (NaN when none is active) */
} rlk_grpo_result_t;

/* Result of rlk_dlogp_audit_ext, written to device memory (all over active tokens). */
typedef struct {
    int64_t active_count;
    int64_t argmax_index;    /* worst token (lowest index on ties); -1 if none is active */
    int64_t argmax_seq;      /* its sequence per seq_offsets; -1 without offsets */
    int64_t argmax_pos;      /* its position inside that sequence; -1 without offsets */
    int64_t clip_count;      /* #{|exp(d) - 1| > clip_eps} */
    double mean_dlogp;       /* mean d */
    double mean_abs_dlogp;   /* mean |d| */
    double mean_ratio;       /* mean ratio0 = mean exp(d) */
    double approx_kl;        /* mean (exp(d) - 1 - d) */
    float max_abs_dlogp;     /* max |d| */
    float p50_abs_dlogp;     /* nearest-rank percentiles of |d|: the value at 1-based rank */
    float p90_abs_dlogp;     /*   ceil(p * count) of the ascending order; exact (radix select) */
    float p99_abs_dlogp;
    float clipfrac;          /* clipfrac0 = clip_count / active_count */
    uint32_t error_flags;    /* bit 0: an active d was not finite */
} rlk_audit_ext_t;

/* Scratch bytes each entry point needs for these sizes (pure arithmetic, no CUDA call). */
size_t rlk_linear_logp_fwd_workspace_bytes(int64_t N, int64_t H, int64_t V);
size_t rlk_linear_logp_bwd_workspace_bytes(int64_t N, int64_t H, int64_t V);
size_t rlk_linear_logp_entropy_bwd_workspace_bytes(int64_t N, int64_t H, int64_t V);
size_t rlk_dlogp_audit_workspace_bytes(int64_t N);
size_t rlk_grpo_clip_loss_workspace_bytes(int64_t N);
size_t rlk_dlogp_audit_ext_workspace_bytes(int64_t N);

/*
 * Forward.  "RL-Kernel Roadmap (2026)" P0.2; "RL-Kernel integration roadmap
 * for vime", linear_logp (the explicit merge of per-block softmax statistics
 * and where the result is downcast).
 *
 *   hidden      [N,H] bf16        weight [V,H] bf16
 *   targets     [N] int64         active_mask [N] uint8 or NULL
 *   temperature T > 0, finite; logits are divided by T before the softmax
 *   logp_out    [N] fp32: logp of active rows, 0 for inactive rows
 *   lse_out     [N] fp32 or NULL: log(sum_v exp(s[t,v]/T)) of active rows,
 *               0 for inactive rows; the backward takes it back
 *   workspace   >= rlk_linear_logp_fwd_workspace_bytes(N, H, V) bytes
 * Logits stay fp32 and are never rounded; logp and lse are fp32.
 */
rlk_status_t rlk_linear_logp_fwd(const void* hidden, const void* weight,
                                 const int64_t* targets, const uint8_t* active_mask,
                                 int64_t N, int64_t H, int64_t V, double temperature,
                                 float* logp_out, float* lse_out,
                                 void* workspace, size_t workspace_bytes,
                                 uint32_t* device_error_word, cudaStream_t stream);

/*
 * Backward by chunked recompute.  "RL-Kernel Roadmap (2026)" P0.2 (the
 * backward recomputes tiles instead of storing logits); "RL-Kernel
 * integration roadmap for vime", linear_logp (dlogits kept as operator-owned
 * workspace, full-gradient training).  With p = softmax(s[t,:]/T) rebuilt
 * from the forward's lse and grad_logp[t] = g_t = dL/dlogp_t:
 *
 *   dhidden[t] = sum_v g_t (delta(v,y_t) - p[t,v]) W_v / T
 *   dweight[v] = sum_t g_t (delta(v,y_t) - p[t,v]) h_t / T
 *
 *   grad_logp  [N] fp32; lse [N] fp32 from rlk_linear_logp_fwd (same inputs)
 *   dhidden    [N,H] bf16 out (0 on inactive rows)
 *   dweight    [V,H] bf16 out, overwritten
 * Accumulation is fp32; dhidden and dweight are rounded to bf16 once (RNE).
 * With an active_mask the GEMMs run over the active rows only (gathered in
 * ascending token order into the workspace): the hidden rows of inactive
 * tokens are never read (NaN padding is harmless), and the result is bit for
 * bit that of the batch made of the active rows alone.
 */
rlk_status_t rlk_linear_logp_bwd(const void* hidden, const void* weight,
                                 const int64_t* targets, const uint8_t* active_mask,
                                 const float* grad_logp, const float* lse,
                                 int64_t N, int64_t H, int64_t V, double temperature,
                                 void* dhidden, void* dweight,
                                 void* workspace, size_t workspace_bytes,
                                 uint32_t* device_error_word, cudaStream_t stream);

/*
 * Forward and backward with the softmax entropy as a second output.
 * "RL-Kernel Roadmap (2026)", backlog: fused entropy / entropy-bonus kernel
 * (next to the fused linear log-prob); "RL-Kernel integration roadmap for
 * vime", linear_logp: entropy requests are served explicitly instead of
 * falling back.  The same tile loop carries one more per-row accumulator,
 * sum_v 2^((s_v - max) k) s_v, so that for active rows
 *
 *   entropy[t] = -sum_v p[t,v] log p[t,v] = lse[t] - E_p[s/T]
 *
 * (fp32; 0 on inactive rows).  Arguments otherwise as rlk_linear_logp_fwd; the
 * workspace query is rlk_linear_logp_fwd_workspace_bytes.  logp and lse equal
 * rlk_linear_logp_fwd's bit for bit.
 */
rlk_status_t rlk_linear_logp_entropy_fwd(const void* hidden, const void* weight,
                                         const int64_t* targets, const uint8_t* active_mask,
                                         int64_t N, int64_t H, int64_t V, double temperature,
                                         float* logp_out, float* lse_out, float* entropy_out,
                                         void* workspace, size_t workspace_bytes,
                                         uint32_t* device_error_word, cudaStream_t stream);

/*
 * Backward of L = sum_t grad_logp[t] logp[t] + sum_t grad_entropy[t] entropy[t],
 * with dentropy/dz_v = -p_v (z_v - E_p[z]) (z = s/T):
 *
 *   dS[t,v] = ( g_t (delta(v,y_t) - p) - gH_t p (z_v - E_p[z]) ) / T
 *
 * lse and entropy are the forward's outputs (E_p[z] = lse - entropy).  Same
 * chunked recompute, rounding and determinism as rlk_linear_logp_bwd, except
 * that dS is kept as two bf16 planes, hi = bf16(dS) and lo = bf16(dS - hi),
 * and the dh and dW GEMMs run over both (twice their K): the entropy gradient
 * has no fp32 part that dominates a row, and one bf16 rounding of dS would
 * cost as much accuracy as the final rounding of the outputs.  Rows with
 * grad_entropy = 0 store lo = 0, so grad_entropy = 0 gives
 * rlk_linear_logp_bwd's dhidden and dweight bit for bit.
 * workspace: rlk_linear_logp_entropy_bwd_workspace_bytes(N, H, V) (the dS
 * part is twice rlk_linear_logp_bwd's).
 */
rlk_status_t rlk_linear_logp_entropy_bwd(const void* hidden, const void* weight,
                                         const int64_t* targets, const uint8_t* active_mask,
                                         const float* grad_logp, const float* grad_entropy,
                                         const float* lse, const float* entropy, int64_t N,
                                         int64_t H, int64_t V, double temperature,
                                         void* dhidden, void* dweight, void* workspace,
                                         size_t workspace_bytes, uint32_t* device_error_word,
                                         cudaStream_t stream);

/*
 * Full-vocabulary KL between the policy head and a reference head (a frozen
 * reference policy, or a teacher for distillation).  "RL-Kernel Roadmap
 * (2026)", backlog: chunked full-vocab KL / distillation KL fused with
 * lm_head, forward and reverse KL over the whole distribution.  For active
 * rows, with p = softmax(hidden W^T / T) and q = softmax(hidden_ref Wr^T / Tr):
 *
 *   kl[t]      = sum_v p[t,v] (log p[t,v] - log q[t,v])        KL(p || q)
 *   kl_rev[t]  = sum_v q[t,v] (log q[t,v] - log p[t,v])        KL(q || p)
 *   lse[t], lse_ref[t]   the two log-partition functions (natural log)
 *   logp[t]    = log p[t, y_t] when targets are given (lse and logp agree with
 *                rlk_linear_logp_fwd's to fp32 rounding)
 *
 * Neither [N,V] logit tensor is materialised: each vocab tile is computed for
 * both heads into the two tensor-memory accumulators and folded into online
 * statistics, merged across 1024-column chunks in ascending order (fixed for
 * a given V: batch invariant).  Inactive rows get 0 everywhere.
 *
 *   hidden [N,H], weight [V,H]; hidden_ref [N,H_ref], weight_ref [V,H_ref]:
 *       bf16, row-major, 16-byte aligned; H and H_ref multiples of 64
 *   targets  [N] int64 or NULL (then logp_out must be NULL)
 *   kl_out   [N] fp32, required; kl_rev_out, lse_out, lse_ref_out, logp_out:
 *       [N] fp32 or NULL
 *   workspace  rlk_linear_kl_fwd_workspace_bytes(N, V) bytes, 256-aligned
 * Errors as rlk_linear_logp_fwd; an active out-of-range target gives logp NaN
 * and RLK_DEVERR_TARGET_RANGE.
 */
size_t rlk_linear_kl_fwd_workspace_bytes(int64_t N, int64_t V);
rlk_status_t rlk_linear_kl_fwd(const void* hidden, const void* weight, const void* hidden_ref,
                               const void* weight_ref, const int64_t* targets,
                               const uint8_t* active_mask, int64_t N, int64_t H, int64_t H_ref,
                               int64_t V, double temperature, double temperature_ref,
                               float* kl_out, float* kl_rev_out, float* lse_out,
                               float* lse_ref_out, float* logp_out, void* workspace,
                               size_t workspace_bytes, uint32_t* device_error_word,
                               cudaStream_t stream);

/*
 * Backward of L = sum_t grad_kl[t] kl[t] + sum_t grad_kl_rev[t] kl_rev[t] with
 * respect to the policy head (the reference head is held fixed):
 *
 *   dS[t,v] = ( g_t p_v (log p_v - log q_v - kl_t) + gr_t (p_v - q_v) ) / T
 *
 * recomputing both heads' logits per tile (chunked like rlk_linear_logp_bwd:
 * dS of one vocab chunk in workspace, fp32 dh accumulation across chunks, no
 * split reductions, no atomics; dh rows batch invariant, dW reproducible bit
 * for bit).  lse, lse_ref and kl are rlk_linear_kl_fwd's outputs; grad_kl or
 * grad_kl_rev may be NULL (not both; kl is needed only with grad_kl).
 * Outputs dhidden [N,H] and dweight [V,H] bf16 (overwritten); inactive rows
 * get dhidden = 0.  Unlike rlk_linear_logp_bwd this backward does not compact
 * a masked batch: the GEMMs run over all N rows, so the hidden rows of
 * inactive tokens (both heads) must hold finite values (a NaN there would
 * reach dweight through 0 * NaN).  As in rlk_linear_logp_entropy_bwd, dS is
 * kept as hi and lo bf16 planes that the dh and dW GEMMs both consume.
 * workspace: rlk_linear_kl_bwd_workspace_bytes(N, H, V)
 * (= rlk_linear_logp_entropy_bwd_workspace_bytes).
 */
size_t rlk_linear_kl_bwd_workspace_bytes(int64_t N, int64_t H, int64_t V);
rlk_status_t rlk_linear_kl_bwd(const void* hidden, const void* weight, const void* hidden_ref,
                               const void* weight_ref, const uint8_t* active_mask,
                               const float* grad_kl, const float* grad_kl_rev, const float* lse,
                               const float* lse_ref, const float* kl, int64_t N, int64_t H,
                               int64_t H_ref, int64_t V, double temperature,
                               double temperature_ref, void* dhidden, void* dweight,
                               void* workspace, size_t workspace_bytes,
                               uint32_t* device_error_word, cudaStream_t stream);

/*
 * Masked dlogp audit.  "RL-Kernel integration roadmap for vime", Consistency
 * Contract: dlogp = recomputed - old over active tokens only; max_abs_dlogp
 * (the primary metric) with the worst-token index; approx_kl0 =
 * mean(exp(dlogp) - 1 - dlogp); active-token count.
 *
 *   logp_new, logp_old [N] fp32; active_mask [N] uint8 or NULL
 *   result_dev  one rlk_audit_result_t in device memory (overwritten)
 *   workspace   rlk_dlogp_audit_workspace_bytes(N) bytes, 256-aligned; its
 *               contents on entry do not matter
 * Fixed-size slices, a fixed assignment of slices to blocks and fixed-order
 * trees: the result is bitwise reproducible for a given N, whatever the
 * inputs' alignment.  Two launches: the per-block partials, then their merge
 * (launched early by programmatic dependent launch).
 */
rlk_status_t rlk_dlogp_audit(const float* logp_new, const float* logp_old,
                             const uint8_t* active_mask, int64_t N,
                             rlk_audit_result_t* result_dev,
                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Vocab-sharded forward, for tensor-parallel LM heads.  "RL-Kernel
 * integration roadmap for vime", linear_logp (TP support: the merge of the
 * vocabulary shards' softmax statistics is an explicit step); "RL-Kernel
 * Roadmap (2026)", TP-invariant reductions.
 *
 * rlk_linear_logp_fwd_shard scores one contiguous block of vocabulary rows
 * [vocab_start, vocab_start + V_local) of the LM head:
 *   weight_shard     [V_local, H] bf16, the block's rows
 *   partials_out     [rlk_linear_logp_num_partials(V_local)][N] pairs of fp32
 *                    (max s, sum_v 2^((s_v - max) log2(e)/T)) per 1024-column
 *                    chunk of the block and row; chunk c of the block is global
 *                    chunk vocab_start/1024 + c
 *   target_logit_out [N] fp32: s[t, y_t] for the rows whose target lies in the
 *                    block; other rows are left untouched
 * vocab_start must be a multiple of 1024 (RLK_ERR_UNSUPPORTED otherwise).
 * rlk_linear_logp_merge then reduces the concatenated partials of all blocks
 * (global chunk order) exactly as rlk_linear_logp_fwd does: when every block
 * but the last holds a multiple of 1024 rows, logp and lse are bitwise equal to
 * the unsharded forward, whatever the number of blocks.  Exchanging the
 * partials between ranks (an all-gather of 8 bytes per row and chunk, plus the
 * target logit from the rank that owns y_t) is the caller's.
 */
int64_t rlk_linear_logp_num_partials(int64_t V_local);
rlk_status_t rlk_linear_logp_fwd_shard(const void* hidden, const void* weight_shard,
                                       const int64_t* targets, const uint8_t* active_mask,
                                       int64_t N, int64_t H, int64_t V_local,
                                       int64_t vocab_start, double temperature,
                                       float* partials_out, float* target_logit_out,
                                       uint32_t* device_error_word, cudaStream_t stream);
/*   partials      [num_partials][N] pairs from rlk_linear_logp_fwd_shard, in global chunk order
 *   num_partials  total over all blocks (= rlk_linear_logp_num_partials(V) when unsharded)
 *   target_logit  [N] fp32, assembled from the owning blocks
 *   V             global vocabulary size (targets outside [0, V) are flagged)
 *   logp_out, lse_out as in rlk_linear_logp_fwd */
rlk_status_t rlk_linear_logp_merge(const float* partials, int64_t num_partials,
                                   const float* target_logit, const int64_t* targets,
                                   const uint8_t* active_mask, int64_t N, int64_t V,
                                   double temperature, float* logp_out, float* lse_out,
                                   uint32_t* device_error_word, cudaStream_t stream);

/*
 * Backward of a vocab-sharded head.  Each block of weight rows [vocab_start,
 * vocab_start + V_local) of a vocab_size-row head contributes
 *
 *   dhidden_partial = sum_{v in block} G[t,v] W_v      (fp32 [N,H], unrounded)
 *   dweight_shard   = rows of dW for the block           (bf16 [V_local,H])
 *
 * with G the logp gradient of rlk_linear_logp_bwd (its fp32 target and
 * dominant-class terms go to the block holding the class).  lse is the
 * merged forward's (rlk_linear_logp_merge); targets are global ids.
 * dweight_shard is bit for bit the matching rows of the unsharded dW (a row's
 * arithmetic does not depend on the blocking).  rlk_linear_logp_dh_merge then
 * sums the partials of all blocks in ascending block order in fp32 and rounds
 * once: dhidden = bf16( sum_r partials[r] ), partial r at dh_partials + r*N*H.
 * Workspace: rlk_linear_logp_bwd_workspace_bytes(N, H, V_local).  The
 * exchange of partials between ranks is the caller's (an all-gather, then the
 * merge in rank order, keeps the result independent of the transport).
 */
rlk_status_t rlk_linear_logp_bwd_shard(const void* hidden, const void* weight_shard,
                                       const int64_t* targets, const uint8_t* active_mask,
                                       const float* grad_logp, const float* lse, int64_t N,
                                       int64_t H, int64_t V_local, int64_t vocab_start,
                                       int64_t vocab_size, double temperature,
                                       float* dhidden_partial, void* dweight_shard,
                                       void* workspace, size_t workspace_bytes,
                                       uint32_t* device_error_word, cudaStream_t stream);
rlk_status_t rlk_linear_logp_dh_merge(const float* dh_partials, int64_t num_partials, int64_t N,
                                      int64_t H, void* dhidden, cudaStream_t stream);

/*
 * Data-parallel gradient exchange of the LM head.  "RL-Kernel Roadmap
 * (2026)", WS2 (a deterministic all-reduce: a fixed rank order with fp32
 * accumulation).  dW sums over the batch, so with the tokens split over
 * ranks every rank holds a partial sum of it; rounding each partial to bf16
 * and summing in whatever order a collective picks would be neither
 * reproducible nor as accurate as one rounding at the end.
 *
 * rlk_linear_logp_bwd_dw_partial is rlk_linear_logp_bwd on one rank's tokens
 * (same arguments, workspace query, dhidden and error behaviour), except that
 * dW is written unrounded:
 *   dweight_partial  [V,H] fp32 (overwritten), 16-byte aligned
 * rlk_linear_logp_dw_merge then forms
 *   dweight = bf16( sum_{r = 0}^{num_partials - 1} dw_partials[r] )   [V,H] bf16
 * with fp32 additions in ascending r (partial r at dw_partials + r*V*H), one
 * RNE rounding per element: the result depends on the partials and their
 * order only.  Gathering the partials in rank order (an all-to-all of row
 * blocks, or an all-gather) is the caller's.  Errors: num_partials < 1, a
 * NULL or unaligned pointer -> RLK_ERR_INVALID_VALUE; H % 64 != 0 ->
 * RLK_ERR_UNSUPPORTED; V = 0 -> RLK_OK, nothing enqueued.
 */
rlk_status_t rlk_linear_logp_bwd_dw_partial(const void* hidden, const void* weight,
                                            const int64_t* targets, const uint8_t* active_mask,
                                            const float* grad_logp, const float* lse, int64_t N,
                                            int64_t H, int64_t V, double temperature,
                                            void* dhidden, float* dweight_partial,
                                            void* workspace, size_t workspace_bytes,
                                            uint32_t* device_error_word, cudaStream_t stream);
rlk_status_t rlk_linear_logp_dw_merge(const float* dw_partials, int64_t num_partials, int64_t V,
                                      int64_t H, void* dweight, cudaStream_t stream);

/*
 * Selected-token logp from existing logits.  "RL-Kernel integration roadmap
 * for vime", logp Reference Scoring: the reference / audit sibling of
 * linear_logp when logits already exist, with the same mask and temperature
 * semantics and a deterministic row-local reduction (fixed topology, fixed
 * launch configuration; dense and indexed rows give identical bits).
 *
 *   logits      [N, row_stride] (V <= row_stride used per row), fp32 or bf16
 *               (dtype = RLK_DTYPE_F32 / RLK_DTYPE_BF16)
 *   rows        [M] int64 row indices to score, or NULL for all N rows (M = N)
 *   targets     [N] int64, active_mask [N] uint8 or NULL (indexed by logits row)
 *   logp_out, lse_out  [M] fp32 (lse_out may be NULL); inactive rows give 0
 * Same arithmetic contract as the fused path: max over raw logits, fp32
 * 2^((x - m) log2(e)/T) sums, lse = (m k + log2 sum) ln 2.  An index outside
 * [0, N) raises RLK_DEVERR_ROW_RANGE and gives NaN for that output.
 */
rlk_status_t rlk_logp_from_logits(const void* logits, int32_t dtype, int64_t N, int64_t V,
                                  int64_t row_stride, const int64_t* rows, int64_t M,
                                  const int64_t* targets, const uint8_t* active_mask,
                                  double temperature, float* logp_out, float* lse_out,
                                  uint32_t* device_error_word, cudaStream_t stream);

/*
 * Fused GRPO / PPO clipped-ratio loss fragment.  "RL-Kernel integration
 * roadmap for vime", RL Loss Operators (fused ratio / loss fragments; the
 * caller owns advantages, clipping range and aggregation); "RL-Kernel Roadmap
 * (2026)", backlog (fused PPO clip loss, ratio-clip-aggregate primitive).
 * For active t, r_t = exp(logp_new[t] - logp_old[t]):
 *
 *   term_t  = min(r_t A_t, clip(r_t, 1 - eps_low, 1 + eps_high) A_t)
 *   loss    = -loss_scale * sum_active term_t
 *   grad[t] = dloss/dlogp_new[t] = -loss_scale A_t r_t where the unclipped
 *             product is the one selected, else 0; 0 on inactive tokens
 *
 *   logp_new, logp_old, advantages [N] fp32; active_mask [N] uint8 or NULL
 *   eps_low, eps_high  >= 0 and finite (eps_low < 1)
 *   loss_scale  > 0 and finite: the aggregation weight, e.g. 1 / (number of
 *               active tokens) for a token mean.  It is the caller's, so each
 *               grad[t] depends on token t alone (batch invariant).
 *   grad_out    [N] fp32, the upstream gradient for rlk_linear_logp_bwd
 *   result_dev  one rlk_grpo_result_t in device memory
 * r and grad are fp32; the sums are fp32 per thread and fp64 across threads
 * in fixed trees (bitwise reproducible for a given N).
 */
rlk_status_t rlk_grpo_clip_loss(const float* logp_new, const float* logp_old,
                                const float* advantages, const uint8_t* active_mask, int64_t N,
                                double eps_low, double eps_high, double loss_scale,
                                float* grad_out, rlk_grpo_result_t* result_dev,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * The consistency contract's minimum diagnostics ("RL-Kernel integration
 * roadmap for vime", Consistency Contract): abs_dlogp mean, max, p50, p90,
 * p99; ratio0 = exp(dlogp); clipfrac0; approx_kl0; active token count; and the
 * worst token's location.  Over active tokens only.
 *
 *   N            <= RLK_AUDIT_EXT_MAX_N (RLK_ERR_UNSUPPORTED above: the
 *                selection counts in 32 bits)
 *   seq_offsets  device int64 [num_seqs + 1] (sequence s holds tokens
 *                [seq_offsets[s], seq_offsets[s+1])), or NULL
 *   clip_eps     >= 0, finite: the ratio0 clip range of clipfrac0
 *   result_dev   one rlk_audit_ext_t in device memory
 * The sums follow rlk_dlogp_audit's fixed blocks and trees; the percentiles
 * are exact order statistics selected with integer histograms, so the whole
 * result is bitwise reproducible for a given N.  ratio0 and the clip test
 * are evaluated in fp32.  The inputs are read once, plus a fixed sample of
 * their 4096-element slices that sets each percentile's window of |d|; a
 * window that misses its rank (a sample unlike the batch) costs two more
 * reads of the inputs, never a different result.
 *
 *   workspace    rlk_dlogp_audit_ext_workspace_bytes(N) bytes (about 12 bytes
 *                per token: room for the candidate lists), 256-aligned; its
 *                contents need not be initialised.  Several launches on
 *                `stream`; calls that share a workspace must not overlap.
 */
#define RLK_AUDIT_EXT_MAX_N ((int64_t)0xffffffff)
rlk_status_t rlk_dlogp_audit_ext(const float* logp_new, const float* logp_old,
                                 const uint8_t* active_mask, int64_t N,
                                 const int64_t* seq_offsets, int64_t num_seqs, double clip_eps,
                                 rlk_audit_ext_t* result_dev, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream);

/*
 * Masked dlogp audit that allocates nothing.  The source pages have no
 * counterpart to this entry point; it exists for callers that cannot call
 * cudaMalloc.  A rollout engine that reserved nearly all device memory for its
 * KV cache at start-up, or a framework hook that may only touch the memory
 * handed to it, can still audit logp without owning a workspace: the scratch
 * lives in a fixed array inside the library.
 *
 * Same inputs, result and arithmetic as rlk_dlogp_audit, minus the workspace.
 *  - N must not exceed RLK_AUDIT_NOALLOC_MAX_N; larger N returns
 *    RLK_ERR_UNSUPPORTED before anything is enqueued (use rlk_dlogp_audit).
 *  - The scratch is a file-scope __device__ array of about 1.25 MiB that
 *    every GPU loading the library holds until the process exits.  Its device
 *    address is looked up on the first call on each device (with that device
 *    current) and again whenever the device's context has been created anew
 *    (after cudaDeviceReset, say); make the first call on a device before any
 *    stream capture.
 *  - Calls share the scratch, which keeps the last call's contents (nothing
 *    in it needs to start at zero: every partial is written before it is
 *    read).  Calls that overlap on the GPU -- on different streams without
 *    ordering -- race and give wrong results.
 *  - No cudaMalloc, cudaFree or other allocating call is made.
 */
#define RLK_AUDIT_NOALLOC_MAX_N ((int64_t)1 << 27)
rlk_status_t rlk_dlogp_audit_noalloc(const float* logp_new, const float* logp_old,
                                     const uint8_t* active_mask, int64_t N,
                                     rlk_audit_result_t* result_dev, cudaStream_t stream);

/* Build fingerprint and the fixed numeric contract (tile shapes, chunk widths,
 * accumulation and rounding points).  Static string, never NULL. */
const char* rlk_contract_string(void);

/* Human-readable name of a status code.  Static string, never NULL. */
const char* rlk_status_string(rlk_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* RLK_H_ */
