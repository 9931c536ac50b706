/*
 * rlk_logp.h -- C ABI of librlk_logp.so: deterministic selected-token
 * log-probability over a tiled vocabulary, on one GB300 GPU (sm_103a).
 *
 * What the library computes (per token row r, real vocabulary V_real):
 *
 *   x_rc     = float(logits[r, c]) for c < V_real; columns c >= V_real are
 *              padding and are masked to -inf before any partial is formed.
 *   tiles    = num_tiles global tiles of width W = V_padded / num_tiles;
 *              tile k covers columns [k*W, (k+1)*W).
 *   partial  = (m_k, s_k) = (max over tile k, sum exp(x - m_k)) in FP32;
 *              a padding-only or all -inf tile is the identity (-inf, 0).
 *   merge    = left fold over k = 0..num_tiles-1 in index order:
 *              m = max(m, m_k), s = s*exp(m_old - m) + s_k*exp(m_k - m).
 *   LSE_r    = m + log s (FP32);  logp_r = x_{r,t_r} - LSE_r (FP32).
 *   dlogits  = g_r * (onehot(t_r) - exp(x_r - LSE_r)) on active rows, BF16,
 *              0 on inactive rows and on padded columns.
 *
 * Sources (pages on the method):
 *   PR #289 "[WS2][PR4][Logp] feat: add distributed TP/CP logprob drift
 *   report": PR-1 commit (typed contract: ShardingSpec with padded-vs-real
 *   vocabulary and owner-rank resolution, MaskSpec, ReductionSpec with an
 *   FP32 (max, sumexp) merge in fixed global index order); commit "docs:
 *   state that cross-TP bitwise equality needs a global tile-level merge
 *   structure" (global tiles, padded columns masked to -inf before the
 *   partials); "typed contract" commit ((-inf, 0) identity partial,
 *   MaskMode explicit_active_mask | ignore_index, FP32 logprob and LSE
 *   outputs, fail-closed dispatch); review excerpt of the vocab-parallel
 *   entry point (tile-size check, active-target validation, non-finite-LSE
 *   error).  Issue #323 "[WS2][Logprob] H100 validation and reproduction
 *   guide", "H100 validation matrix" (BF16 logits, FP32 accumulation,
 *   bitwise-identical outputs across TP degrees).  The H100 matrix
 *   document "H100 canonical TP/CP validation", "Fixes exercised" (fixed
 *   virtual TP8 and vocabulary 152576).
 *
 * Conventions for every entry point:
 *   - Device pointers are CUDA global-memory pointers owned by the caller;
 *     the library allocates nothing and keeps no pointer after returning.
 *     Every pointer must be device (or managed) memory of the device that
 *     holds the call's first operand; host memory, pinned or not, and
 *     another GPU's memory return RLK_ERR_INVALID_ARG before any launch.
 *   - Work is enqueued on `stream` (NULL = the legacy default stream) and
 *     is asynchronous, unless contract->validate == 1: then the call
 *     synchronises the stream and turns the device status word into the
 *     return code.
 *   - Errors are status codes; nothing throws or exits.  A contract the
 *     kernels do not support returns RLK_ERR_UNSUPPORTED -- there is no
 *     fallback of any kind.  rlk_last_error_message() gives the reason
 *     (per calling thread).
 *   - Results do not depend on virtual_tp: outputs are bitwise identical
 *     for virtual_tp = 1, 2, 4, 8.
 */
#ifndef RLK_LOGP_H
#define RLK_LOGP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st* rlk_stream_t;

typedef enum {
    RLK_OK = 0,
    RLK_ERR_INVALID_ARG = 1,   /* null/inconsistent pointer or field */
    RLK_ERR_UNSUPPORTED = 2,   /* well-formed but outside what the kernels do; fail closed */
    RLK_ERR_NON_TILEABLE = 3,  /* num_tiles does not divide V_padded, or virtual_tp does not divide num_tiles */
    RLK_ERR_MISALIGNED = 4,    /* a pointer or the row stride is not 16-byte aligned */
    RLK_ERR_TARGET_RANGE = 5,  /* an active target outside [0, V_real) (device status) */
    RLK_ERR_NONFINITE_LSE = 6, /* an active row's LSE is not finite (device status) */
    RLK_ERR_TIMEOUT = 7,       /* a bounded device-side wait expired (device status) */
    RLK_ERR_CUDA = 8           /* a CUDA runtime call failed, or (device status) a streaming kernel found a ring
                                  slot holding an unexpected row and stopped before touching memory */
} rlk_status;

typedef enum {
    RLK_MASK_EXPLICIT = 0,     /* active_mask[r] != 0 marks an active row; targets of inactive rows are never read as indices */
    RLK_MASK_IGNORE_INDEX = 1  /* a row is active iff targets[r] != ignore_index; active_mask must be NULL */
} rlk_mask_mode;

/*
 * The contract (PR #289, PR-1 and "typed contract" commits: LogprobContract,
 * ShardingSpec, MaskSpec, ReductionSpec).  64 bytes, no padding.
 */
typedef struct {
    int64_t T;               /* token rows, >= 0 */
    int64_t V_real;          /* real vocabulary, >= 1; columns >= V_real are padding */
    int64_t V_padded;        /* padded vocabulary, >= V_real; num_tiles must divide it */
    int64_t row_stride;      /* elements between rows of logits and of dlogits; 0 -> V_padded;
                                must be >= V_padded and a multiple of 8 (16-byte rows) */
    int32_t num_tiles;       /* global vocabulary tiles (64 in the pages' runs); 1..1024,
                                tile width V_padded/num_tiles at most 16384 */
    int32_t virtual_tp;      /* 1, 2, 4 or 8 vocabulary shards (tile-aligned, must divide num_tiles) */
    int32_t mask_mode;       /* rlk_mask_mode */
    int32_t validate;        /* 0: asynchronous; 1: synchronise and report device status */
    int64_t ignore_index;    /* RLK_MASK_IGNORE_INDEX only (the pages use -100) */
    int64_t wait_timeout_ns; /* bound of every device-side wait; 0 -> 2 s */
} rlk_logp_contract;

/*
 * Host-only validation of a contract (PR #289 review excerpt: _tile_size and
 * _validate_invocation run before any work).  Touches no device.
 * Returns RLK_OK, RLK_ERR_INVALID_ARG, RLK_ERR_NON_TILEABLE,
 * RLK_ERR_MISALIGNED or RLK_ERR_UNSUPPORTED.
 */
rlk_status rlk_logp_check_contract(const rlk_logp_contract* contract);

/*
 * Bytes of device workspace rlk_logp_fwd / rlk_logp_bwd need (the device
 * status word); 0 for an invalid contract.  The workspace must be 16-byte
 * aligned and must not be shared by calls that may run concurrently.
 */
size_t rlk_logp_workspace_size(const rlk_logp_contract* contract);

/*
 * Forward: LSE and selected log-probability of every row.
 *   logits_bf16  [T, row_stride] BF16, row-major, 16-byte aligned; only
 *                columns < V_real are read.
 *   targets      [T] int64.  Active targets must lie in [0, V_real).
 *   active_mask  [T] uint8 (RLK_MASK_EXPLICIT), or NULL (RLK_MASK_IGNORE_INDEX).
 *   logp         [T] FP32 out: x_t - LSE on active rows, +0.0 on inactive rows,
 *                NaN on an active row whose target is out of range.
 *   lse          [T] FP32 out: LSE of every row (active or not).
 *   partials     NULL, or [T, num_tiles, 2] FP32 out: the (m_k, s_k) partials.
 *   workspace    rlk_logp_workspace_size() bytes.
 * Device status: RLK_ERR_TARGET_RANGE for an active target outside
 * [0, V_real); RLK_ERR_NONFINITE_LSE for an active row with a non-finite LSE
 * (PR #289 review excerpt: "non-finite logsumexp on an active row").
 */
rlk_status rlk_logp_fwd(const rlk_logp_contract* contract, const void* logits_bf16,
                        const int64_t* targets, const uint8_t* active_mask, float* logp,
                        float* lse, float* partials, void* workspace, rlk_stream_t stream);

/*
 * Forward plus the entropy of each row's softmax over the real vocabulary,
 * in the same single pass over the logits: every tile also sums
 * t_k = sum_c e^(x_c - m_k) x_c beside s_k, the fold runs the same
 * fixed-order recurrence on it, and entropy = LSE - (sum_c p_c x_c), which
 * equals -sum_c p_c log p_c.  The pages log a mean policy entropy beside the
 * loss in their RL runs (the H100 matrix document, "Completed full-model
 * matrix"); the formula is Shannon's.
 *   entropy      [T] FP32 out, every row (active or not); NaN where the LSE
 *                is not finite.
 * Every other argument, output and status is that of rlk_logp_fwd; logp and
 * LSE are bitwise those of rlk_logp_fwd.  Outputs are bitwise identical for
 * every virtual_tp.
 */
rlk_status rlk_logp_fwd_entropy(const rlk_logp_contract* contract, const void* logits_bf16,
                                const int64_t* targets, const uint8_t* active_mask, float* logp, float* lse,
                                float* entropy, void* workspace, rlk_stream_t stream);

/*
 * The fused single-pass forward+backward (rlk_logp_bwd with lse_in == NULL)
 * plus the entropy of each row's softmax, as rlk_logp_fwd_entropy computes
 * it, in the same pass over the logits: the step of RL training that also
 * logs the policy's entropy.  dlogits, logp_out and lse_out are bitwise
 * those of rlk_logp_bwd; entropy_out ([T] FP32, every row, NaN where the LSE
 * is not finite) is bitwise that of rlk_logp_fwd_entropy.  Every argument is
 * required; row_stride, masks, status and in-place dlogits as for
 * rlk_logp_bwd.  Runs the L2 fused schedule (RLK_FUSED_SCHEDULE=resident
 * returns RLK_ERR_UNSUPPORTED).
 */
rlk_status rlk_logp_fwd_bwd_entropy(const rlk_logp_contract* contract, const void* logits_bf16,
                                    const int64_t* targets, const uint8_t* active_mask, const float* grad_logp,
                                    void* dlogits_bf16, float* logp_out, float* lse_out, float* entropy_out,
                                    void* workspace, rlk_stream_t stream);

/*
 * Token-mean GRPO loss of per-token log-probabilities and its gradient with
 * respect to each logp: the step after the forward, whose g feeds
 * rlk_logp_bwd.  The pages name a GRPO loss contract (issue #323 "[WS2]
 * [Logprob] H100 validation and reproduction guide", "Validation Boundary":
 * the PR5 GRPO contract tests) and a KL coefficient of 0.01 (the H100 matrix
 * document, "Completed full-model matrix") but print no formula; this is the
 * convention:
 *   N     = number of active rows (token mean); with N = 0 the loss and every
 *           gradient are 0;
 *   loss  = (1/N) sum over active r of (-A_r logp_r + beta k3_r), where
 *           k3_r = exp(ref_r - logp_r) - (ref_r - logp_r) - 1 if ref_logp is
 *           given (the k3 estimator of KL(pi || pi_ref)), else no KL term;
 *   g_r   = (mask_r / N) (-A_r + beta (1 - exp(ref_r - logp_r))).
 * Arguments (device pointers, FP32 unless said): logp, advantage (per row;
 * a caller broadcasts per-sequence advantages), active_mask (uint8), ref_logp
 * (NULL: no KL term), beta (>= 0), loss (one float out), grad_logp ([T] out),
 * active_count (NULL, or one float out: N, exact up to 2^24).  Per-row terms
 * are FP32; one cluster of 8 CTAs sums them in FP64 in a fixed order that
 * depends on T only, so the loss is bitwise reproducible.  grad_logp must not
 * overlap the inputs.  Asynchronous on `stream`; returns RLK_ERR_INVALID_ARG
 * for missing pointers or a bad beta.
 */
rlk_status rlk_grpo_loss(int64_t T, const float* logp, const float* advantage, const uint8_t* active_mask,
                         const float* ref_logp, float beta, float* loss, float* grad_logp, float* active_count,
                         rlk_stream_t stream);

/*
 * The GRPO training step of the logits in one pass over them: logp, LSE,
 * the GRPO loss, its gradient g and dlogits = g (onehot - softmax), with or
 * without the KL term.  rlk_grpo_loss's g depends on logp, so composed from
 * the calls above the step needs rlk_logp_fwd, rlk_grpo_loss, then
 * rlk_logp_bwd with lse_in (the logits read twice).  Here each row's g is
 * formed on chip as soon as the fused pass has the row's logp, by exactly
 * the operations rlk_grpo_loss uses, and the row's dlogits follow at once.
 * The loss, g, logp, LSE and dlogits are bitwise those of that composition.
 *   contract      as for rlk_logp_bwd (either mask mode); runs the L2 fused
 *                 schedule (RLK_FUSED_SCHEDULE=resident: RLK_ERR_UNSUPPORTED).
 *   advantage     [T] FP32, per row (broadcast per-sequence values).
 *   ref_logp      [T] FP32, or NULL for no KL term; beta >= 0 as for
 *                 rlk_grpo_loss.  N = the contract's active rows.
 *   dlogits_bf16  [T, row_stride] out, as for rlk_logp_bwd; may be the
 *                 logits themselves (in place).
 *   logp_out, lse_out, grad_out  [T] FP32 out (grad_out: g of every row).
 *   entropy_out   [T] FP32 out, or NULL: the entropy of each row's softmax
 *                 (bitwise rlk_logp_fwd_entropy's).
 *   loss          one FP32 out; active_count NULL or one FP32 out (N).
 *   workspace     rlk_grpo_fused_workspace_size bytes.
 * The loss convention and its sources on the pages are rlk_grpo_loss's
 * (above).  T = 0 writes loss = 0 (and N = 0).  Host checks return
 * RLK_ERR_INVALID_ARG for a missing pointer, a negative or non-finite beta,
 * or dlogits overlapping the logits other than exactly; device status as for
 * rlk_logp_bwd.  The workspace belongs to one call at a time.
 */
size_t rlk_grpo_fused_workspace_size(const rlk_logp_contract* contract);
rlk_status rlk_grpo_fused_step(const rlk_logp_contract* contract, const void* logits_bf16, const int64_t* targets,
                               const uint8_t* active_mask, const float* advantage, const float* ref_logp,
                               float beta, void* dlogits_bf16, float* logp_out, float* lse_out, float* grad_out,
                               float* entropy_out, float* loss, float* active_count, void* workspace,
                               rlk_stream_t stream);

/*
 * Backward (and, with lse_in == NULL, the fused single-pass forward+backward).
 *   grad_logp    [T] FP32: upstream gradient g_r of logp_r (used on active rows).
 *   dlogits_bf16 [T, row_stride] BF16 out, 16-byte aligned: columns
 *                [0, V_padded) of every row are written (padding and inactive
 *                rows exactly 0); columns >= V_padded are not touched.
 *   lse_in       [T] FP32 from an earlier rlk_logp_fwd, or NULL.  With
 *                lse_in != NULL the logits are re-read and logp_out/lse_out
 *                must be NULL.  With lse_in == NULL each logits row is read
 *                once: LSE is formed on chip, dlogits written, and
 *                logp_out/lse_out (both required) receive the forward
 *                outputs, bitwise equal to rlk_logp_fwd's.
 * dlogits are bitwise identical between the two forms.  The fused form
 * reads each row's bytes from HBM once and its second copy from L2 (any
 * vocabulary); RLK_FUSED_SCHEDULE=resident instead keeps a row's slice in
 * shared memory across a cluster of CTAs and returns RLK_ERR_UNSUPPORTED for
 * a vocabulary too large for that.
 * In place: dlogits_bf16 may be logits_bf16 itself (the same pointer and
 * row_stride), in both forms -- every logit is read before its gradient
 * overwrites it, and the outputs are bitwise those of a separate buffer.
 * Any other overlap of an output with an input is not allowed.
 */
rlk_status rlk_logp_bwd(const rlk_logp_contract* contract, const void* logits_bf16,
                        const int64_t* targets, const uint8_t* active_mask,
                        const float* lse_in, const float* grad_logp, void* dlogits_bf16,
                        float* logp_out, float* lse_out, void* workspace, rlk_stream_t stream);

/*
 * Bytes of device workspace every fused lm_head call (rlk_logp_fused_lmhead
 * and the _bwd, _keep and _bwd_kept forms) needs for hidden size H: the status word, 256 bytes of work tickets, FP32
 * partials [T, num_tiles * ceil(V_padded / num_tiles / 256), 2] (one per
 * 256-row weight chunk), target logits [T], and for the backward the BF16
 * dlogits [T, V_padded] and the forward's FP32 logits [T, V_padded] (about
 * T * V_padded * 6 bytes in all: 7.5 GB for 8192 x 152576); 0 for an
 * unsupported contract.
 */
size_t rlk_logp_lmhead_workspace_size(const rlk_logp_contract* contract, int64_t H);

/*
 * Fused lm_head: logp and LSE of logits = hidden @ weight^T without
 * materialising the logits (the optional fused kernel of issue #323,
 * "Validation Boundary").  A tcgen05 GEMM (FP32 accumulators in tensor
 * memory) turns each (128-token block, 256-row weight chunk) into the chunk's
 * (max, sumexp) partial in its epilogue; a tile's chunks are merged in chunk
 * order and the tiles folded in fixed tile order.  The logits stay FP32
 * (never rounded to BF16).
 *   hidden_bf16  [T, H] BF16 row-major, 16-byte aligned; H a multiple of 64.
 *   weight_bf16  [V_padded, H] BF16 row-major; rows >= V_real are padding
 *                and are never read.
 *   targets, active_mask, logp, lse: as for rlk_logp_fwd.
 *   grad_logp    NULL (forward only) or [T] FP32 upstream gradient of logp.
 *                With it the backward runs too: the forward also writes its
 *                FP32 logits to the workspace, an elementwise pass forms
 *                dlogits = g (onehot - softmax) from them and the LSE just
 *                formed (BF16, in the workspace), then two more tcgen05 GEMMs
 *                with FP32 accumulation give
 *   dhidden_bf16 [T, H] BF16 out = dlogits[:, :V_real] @ weight[:V_real], and
 *   dweight_f32  [V_padded, H] FP32 out, or NULL, and
 *   dweight_bf16 [V_padded, H] BF16 out, or NULL (at least one of the two):
 *                dlogits[:, :V_real]^T @ hidden, rows >= V_real exactly 0.
 *                Each output element is accumulated over its whole K range in
 *                one fixed order by one CTA (no split-K, no atomics), so the
 *                gradients are deterministic.  All three NULL without grad_logp.
 *   workspace    rlk_logp_lmhead_workspace_size(contract, H) bytes (for the
 *                backward it holds the FP32 logits and the BF16 dlogits,
 *                T * V_padded * 6 bytes).
 * The tile width V_padded / num_tiles must be a multiple of 16.  row_stride
 * is not used.  Outputs are bitwise identical for every virtual_tp.
 */
rlk_status rlk_logp_fused_lmhead(const rlk_logp_contract* contract, const void* hidden_bf16, int64_t H,
                                 const void* weight_bf16, const int64_t* targets, const uint8_t* active_mask,
                                 const float* grad_logp, float* logp, float* lse, void* dhidden_bf16,
                                 float* dweight_f32, void* dweight_bf16, void* workspace, rlk_stream_t stream);

/*
 * The fused lm_head backward alone, from the LSE an earlier forward returned
 * (rlk_logp_fused_lmhead without grad_logp): the recompute GEMM writes
 * dlogits = g (onehot - exp(x - lse_in)) in BF16, then the dHidden and dW
 * GEMMs run, exactly as in rlk_logp_fused_lmhead with grad_logp (so the
 * outputs are bitwise those of that call when lse_in is its LSE).  It skips
 * the forward GEMM: an autograd backward costs three GEMM passes, not four.
 *   lse_in      [T] FP32; grad_logp [T] FP32; the other arguments and
 *               outputs as for rlk_logp_fused_lmhead.
 * Device status (validate == 1): an active target outside [0, V_real), a
 * non-finite lse_in on an active row.
 */
rlk_status rlk_logp_fused_lmhead_bwd(const rlk_logp_contract* contract, const void* hidden_bf16, int64_t H,
                                     const void* weight_bf16, const int64_t* targets, const uint8_t* active_mask,
                                     const float* lse_in, const float* grad_logp, void* dhidden_bf16,
                                     float* dweight_f32, void* dweight_bf16, void* workspace, rlk_stream_t stream);

/*
 * The fused lm_head forward that also keeps its FP32 logits for a later
 * backward, for an autograd forward that trades T * V_padded * 4 bytes, held
 * until the backward, for the backward's recompute GEMM (the split form of
 * what rlk_logp_fused_lmhead with grad_logp does inside one call).
 *   logits_f32  [T, V_padded] FP32 out, 16-byte aligned, written in full:
 *               hidden @ weight^T as the GEMM accumulated it (columns >= V_real
 *               hold products with the padding rows and are never used).
 *   the other arguments and outputs as for rlk_logp_fused_lmhead without
 *   grad_logp; logp and lse are bitwise those of that call.
 */
rlk_status rlk_logp_fused_lmhead_keep(const rlk_logp_contract* contract, const void* hidden_bf16, int64_t H,
                                      const void* weight_bf16, const int64_t* targets, const uint8_t* active_mask,
                                      float* logp, float* lse, float* logits_f32, void* workspace,
                                      rlk_stream_t stream);

/*
 * The fused lm_head backward from the logits rlk_logp_fused_lmhead_keep kept
 * and its LSE: an HBM-bound pass writes dlogits = g (onehot - exp(x - lse_in))
 * in BF16, then the dHidden and dW GEMMs run.  The outputs are bitwise those
 * of rlk_logp_fused_lmhead_bwd with the same lse_in, and of
 * rlk_logp_fused_lmhead with grad_logp.
 *   logits_f32  [T, V_padded] FP32 in, 16-byte aligned, as the forward wrote
 *               it; not modified.
 *   the other arguments and outputs as for rlk_logp_fused_lmhead_bwd; no
 *   output may overlap an input.
 * Device status (validate == 1): as for rlk_logp_fused_lmhead_bwd.
 */
rlk_status rlk_logp_fused_lmhead_bwd_kept(const rlk_logp_contract* contract, const void* hidden_bf16, int64_t H,
                                          const void* weight_bf16, const int64_t* targets,
                                          const uint8_t* active_mask, const float* lse_in, const float* logits_f32,
                                          const float* grad_logp, void* dhidden_bf16, float* dweight_f32,
                                          void* dweight_bf16, void* workspace, rlk_stream_t stream);

/*
 * Vocabulary-parallel tensor parallelism across GPUs (PR #289 "[WS2][PR4]
 * [Logp] feat: add distributed TP/CP logprob drift report", PR-1 contract
 * commit: tile-aligned vocabulary shards, FP32 (max, sumexp) partials moved by
 * all-gather and merged by every rank in fixed global tile order, the target
 * logit taken from the owner rank; issue #323, "Six-Case TP/CP Matrix").
 * The three calls below are what one rank runs; the exchange between them is
 * the caller's all-gather (NCCL, say) of plain device buffers.
 *
 * A shard call's contract is the whole problem's: T, V_real, V_padded,
 * num_tiles, mask mode, ignore_index as for rlk_logp_fwd, and virtual_tp =
 * tp, the number of shards (1, 2, 4 or 8, dividing num_tiles).  Shard j
 * holds columns [j*Vs, (j+1)*Vs) of the padded vocabulary, Vs = V_padded/tp,
 * which must be a multiple of 8 (16-byte shard starts), in a buffer of its
 * own: logits_shard [T, row_stride] BF16 with row_stride >= Vs (0 -> Vs), a
 * multiple of 8.  Targets are global column indices.  The results are
 * bitwise those of rlk_logp_fwd / rlk_logp_bwd on the whole vocabulary, for
 * every tp.
 */

/* Host-only check of a shard call's contract and shard index (touches no device). */
rlk_status rlk_logp_check_shard_contract(const rlk_logp_contract* contract, int32_t shard);

/* Bytes of device workspace each shard call needs; 0 for an invalid contract. */
size_t rlk_logp_shard_workspace_size(const rlk_logp_contract* contract);

/*
 * Rank side of the forward, on shard `shard`:
 *   partials_shard [T, num_tiles/tp, 2] FP32 out: the (m_k, s_k) partials of
 *                  global tiles shard*num_tiles/tp .. (shard+1)*num_tiles/tp - 1;
 *   target_logit   [T] FP32 out: float(logit[r, t_r]) on active rows whose
 *                  target column this shard holds, 0 on every other row.
 * No target is checked here (the fold does).
 */
rlk_status rlk_logp_shard_fwd(const rlk_logp_contract* contract, int32_t shard, const void* logits_shard,
                              const int64_t* targets, const uint8_t* active_mask, float* partials_shard,
                              float* target_logit, void* workspace, rlk_stream_t stream);

/*
 * The merge after the exchange, run by every rank on the same gathered data:
 *   gathered_partials     [tp, T, num_tiles/tp, 2] FP32: every shard's
 *                         partials_shard, shard-major (what an all-gather of
 *                         them along a new leading dimension leaves);
 *   gathered_target_logit [tp, T] FP32: every shard's target_logit.
 *   logp, lse             [T] FP32 out, as rlk_logp_fwd's (the target logit
 *                         is taken from shard t_r / Vs).
 * Device status as for rlk_logp_fwd (target range, non-finite LSE).
 */
rlk_status rlk_logp_fold(const rlk_logp_contract* contract, const float* gathered_partials,
                         const float* gathered_target_logit, const int64_t* targets, const uint8_t* active_mask,
                         float* logp, float* lse, void* workspace, rlk_stream_t stream);

/*
 * Rank side of the backward, given the (replicated) LSE from rlk_logp_fold:
 *   dlogits_shard [T, row_stride] BF16 out: columns [0, Vs) of every row,
 *                 g (onehot - exp(x - LSE)) with the one-hot term only in the
 *                 shard that holds the target; padding and inactive rows 0.
 * No collective is needed.  dlogits_shard may be logits_shard itself (in
 * place, as for rlk_logp_bwd).  Device status: an active target outside
 * [0, V_real), a non-finite lse_in on an active row.
 */
rlk_status rlk_logp_shard_bwd(const rlk_logp_contract* contract, int32_t shard, const void* logits_shard,
                              const int64_t* targets, const uint8_t* active_mask, const float* lse_in,
                              const float* grad_logp, void* dlogits_shard, void* workspace, rlk_stream_t stream);

/*
 * rlk_logp_fwd without a workspace argument, for callers that cannot
 * allocate device memory while they run: an engine or server whose device
 * memory is reserved up front, a plugin that is handed a stream but no
 * allocator, or a step that must not call the synchronising cudaMalloc.
 * (The pages have no counterpart; this entry point only changes where the
 * scratch lives.)
 *
 * Arguments and results are those of rlk_logp_fwd.  The forward's scratch --
 * the status word, at most 256 bytes -- lives in a static device array that
 * every GPU which loads the library holds until the process exits; a contract
 * that would need more returns RLK_ERR_UNSUPPORTED.  The call allocates no
 * device memory and calls no allocating routine.  The first call on a device
 * looks up the array's device address with that device current (one
 * cudaGetSymbolAddress); make that first call before any stream capture.
 * The address is kept per device together with the id of the CUDA context
 * it was looked up in; if that context is gone (cudaDeviceReset, say), the
 * next call looks the address up again in the new context, so make the
 * first call after a reset before any stream capture too.
 * Every call on a device shares the one array and clears the status word
 * first, so calls that overlap on the GPU race on it: serialise them (one
 * stream, or events).  Device-side conditions (RLK_ERR_TARGET_RANGE,
 * RLK_ERR_NONFINITE_LSE, RLK_ERR_TIMEOUT) are returned only with
 * validate == 1; with validate == 0 the call is asynchronous and they are
 * not reported (an out-of-range active target still yields logp = NaN).
 */
rlk_status rlk_logp_fwd_noalloc(const rlk_logp_contract* contract, const void* logits_bf16,
                                const int64_t* targets, const uint8_t* active_mask, float* logp,
                                float* lse, float* partials, rlk_stream_t stream);

/*
 * Synchronises `stream` and decodes the status word a previous asynchronous
 * call left in `workspace` (RLK_OK when no device-side error was recorded).
 */
rlk_status rlk_logp_workspace_status(const void* workspace, rlk_stream_t stream);

/*
 * Self-test of the kernels' bounded device-side waits: one warp waits, with
 * the same code the kernels use, on an mbarrier that nothing arrives at.
 * The wait expires after timeout_ns (0 < timeout_ns <= 10 s), records the
 * timeout in the status word and the kernel returns; the call synchronises
 * `stream` and returns RLK_ERR_TIMEOUT when the mechanism works.  Nothing
 * faults and the context stays usable.  `workspace` as for rlk_logp_fwd.
 * (A check of the failure-detection path; the pages have no counterpart.)
 */
rlk_status rlk_selftest_bounded_wait(int64_t timeout_ns, void* workspace, rlk_stream_t stream);

/* Static text of a status code. */
const char* rlk_status_string(rlk_status status);

/* Reason for the last non-OK return on the calling thread ("" if none). */
const char* rlk_last_error_message(void);

#ifdef __cplusplus
}
#endif

#endif /* RLK_LOGP_H */
