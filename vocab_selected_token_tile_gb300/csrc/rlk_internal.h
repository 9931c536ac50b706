// Internal declarations shared by the C ABI (rlk_api.cu) and the kernels'
// launch planners.  Not part of the public interface.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "rlk_logp.h"

namespace rlk {

// Device status word bits (written by kernels with atomicOr, read by the host).
enum : uint32_t {
    kStatusTargetRange = 1u << 0,
    kStatusNonFinite = 1u << 1,
    kStatusTimeout = 1u << 2,
    kStatusInternal = 1u << 3,  // a kernel found its own bookkeeping inconsistent and stopped
};

constexpr int kMaxTiles = 1024;
constexpr int64_t kMaxTileCols = 16384;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;  // 2 s
constexpr size_t kWorkspaceBytes = 256;

// kModeFused is what callers ask for; the planner runs it as kModeFusedL2
// (second read of each row from L2) unless RLK_FUSED_SCHEDULE=resident.
enum StreamMode : int { kModeFwd = 0, kModeBwd = 1, kModeFused = 2, kModeFusedL2 = 3 };

// Arguments of one streaming launch (all device pointers).
struct StreamArgs {
    const uint16_t* logits;
    uint16_t* dlogits;
    const int64_t* targets;
    const uint8_t* mask;
    const float* grad;
    const float* lse_in;
    float* logp;
    float* lse;
    float* partials;
    float* entropy;  // optional (forward): entropy of each row's softmax
    uint32_t* status;
    // kModeBwd on one vocabulary shard: an active row's target may lie in
    // another shard (any value outside [0, V_real) of this launch); it then
    // takes no one-hot term here and is not an error.
    int32_t foreign_targets;
    // The fused GRPO step (kModeFusedL2): instead of reading g, each row's g
    // is formed on chip from its logp once the fold has it,
    //   g_r = mask_r (-A_r + beta (1 - exp(ref_r - logp_r))) / N
    // (no KL term without ref), in the same FP32 operations as the GRPO loss
    // kernel, and written to grad_out.  n_active holds N.
    int32_t grpo;
    const float* adv;
    const float* ref;
    float beta;
    const unsigned long long* n_active;
    float* grad_out;
};

// Records a failure reason for rlk_last_error_message() and returns `s`.
rlk_status fail(rlk_status s, const std::string& why);

// Host check of the planner overrides in the environment (RLK_CTAS_PER_SM,
// RLK_ROW_BUFS, RLK_FUSED_SKEW, RLK_FUSED_SCHEDULE): RLK_ERR_UNSUPPORTED for
// any value outside the ring shapes the protocol model replays.
rlk_status check_planner_env();

// Launches one streaming kernel (mode kModeFwd / kModeBwd / kModeFused) for a
// validated contract; returns RLK_OK or an error with the message set.
rlk_status launch_stream(const rlk_logp_contract& c, int mode, const StreamArgs& a, cudaStream_t stream);

// Fused lm_head (lmhead.cu): host checks, workspace bytes beyond the status
// area, and the forward launch (GEMM + epilogue partials, then the fold).
rlk_status lmhead_check(const rlk_logp_contract& c, int64_t H);
size_t lmhead_fwd_workspace(const rlk_logp_contract& c);
rlk_status launch_lmhead_fwd(const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                             const int64_t* targets, const uint8_t* mask, float* logp, float* lse, void* workspace,
                             uint32_t* status, cudaStream_t stream);

size_t lmhead_bwd_workspace(const rlk_logp_contract& c);
rlk_status launch_lmhead_bwd(const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                             const int64_t* targets, const uint8_t* mask, const float* grad, float* logp, float* lse,
                             void* dhidden, float* dweight_f32, void* dweight_bf16, void* workspace, uint32_t* status,
                             cudaStream_t stream);
// The forward that also writes its FP32 logits [T, V_padded] to logits_f32.
rlk_status launch_lmhead_fwd_keep(const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                                  const int64_t* targets, const uint8_t* mask, float* logp, float* lse,
                                  float* logits_f32, void* workspace, uint32_t* status, cudaStream_t stream);
// The backward from kept FP32 logits and the LSE: dlogits pass, then dHidden and dW.
rlk_status launch_lmhead_bwd_kept(const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                                  const int64_t* targets, const uint8_t* mask, const float* grad, const float* lse,
                                  const float* logits_f32, void* dhidden, float* dweight_f32, void* dweight_bf16,
                                  void* workspace, uint32_t* status, cudaStream_t stream);
// The backward alone, from a given LSE: recompute GEMM (dlogits), then dHidden and dW.
rlk_status launch_lmhead_bwd_given_lse(const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                                       const int64_t* targets, const uint8_t* mask, const float* grad,
                                       const float* lse, void* dhidden, float* dweight_f32, void* dweight_bf16,
                                       void* workspace, uint32_t* status, cudaStream_t stream);

// Vocabulary-parallel pieces (shard.cu).  A shard call's contract describes
// the whole problem with virtual_tp = the number of shards; shard j holds
// columns [j*Vs, (j+1)*Vs) of the padded vocabulary, Vs = V_padded/virtual_tp.
rlk_status check_shard_contract(const rlk_logp_contract& c, int32_t shard);
// The contract of shard j's columns as a vocabulary of its own (V_real of it
// may be 0: a shard of padding only).
rlk_logp_contract shard_local_contract(const rlk_logp_contract& c, int32_t shard);
size_t shard_workspace(const rlk_logp_contract& c);
rlk_status launch_shard_fwd(const rlk_logp_contract& c, int32_t shard, const uint16_t* logits, const int64_t* targets,
                            const uint8_t* mask, float* partials, float* target_logit, void* workspace,
                            uint32_t* status, cudaStream_t stream);
rlk_status launch_gathered_fold(const rlk_logp_contract& c, const float* gathered_partials,
                                const float* gathered_xt, const int64_t* targets, const uint8_t* mask, float* logp,
                                float* lse, uint32_t* status, cudaStream_t stream);
rlk_status launch_shard_bwd(const rlk_logp_contract& c, int32_t shard, const uint16_t* logits, const int64_t* targets,
                            const uint8_t* mask, const float* lse_in, const float* grad, uint16_t* dlogits,
                            void* workspace, uint32_t* status, cudaStream_t stream);

// Token-mean GRPO loss and its gradient (grpo_loss.cu); one cluster, fixed
// order.  grad may be NULL (the loss alone).
rlk_status launch_grpo_loss(int64_t T, const float* logp, const float* adv, const uint8_t* mask, const float* ref,
                            float beta, float* loss, float* grad, float* count, cudaStream_t stream);

// N of the fused GRPO step into *n_active (cleared first); in ignore_index
// mode (mask NULL) each row's activity also goes to mask_out.
rlk_status launch_grpo_count(int64_t T, const int64_t* targets, const uint8_t* mask, int64_t ignore_index,
                             uint8_t* mask_out, unsigned long long* n_active, int sm_count, cudaStream_t stream);

// Launches the bounded-wait self-test kernel (one warp waiting on an mbarrier
// that nothing arrives at).
rlk_status launch_selftest_wait(uint64_t limit_ns, uint32_t* status, cudaStream_t stream);

}  // namespace rlk
