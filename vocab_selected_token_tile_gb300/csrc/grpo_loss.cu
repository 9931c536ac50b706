// Token-mean GRPO loss of per-token log-probabilities and its gradient with
// respect to each logp (sm_103a).
//
// The pages name a GRPO loss contract (issue #323 "[WS2][Logprob] H100
// validation and reproduction guide", "Validation Boundary": the PR5 GRPO
// contract tests) and run it with a KL coefficient of 0.01 (the H100 matrix
// document, "Completed full-model matrix"), but print no formula.  The
// convention, stated in full:
//   N      = active tokens of the batch (token mean); with N = 0 the loss and
//            every gradient are 0;
//   loss   = (1/N) sum over active r of (-A_r logp_r + beta k3_r),
//            k3_r = exp(ref_r - logp_r) - (ref_r - logp_r) - 1 when a
//            reference logp is given (else no KL term);
//   g_r    = (mask_r / N) (-A_r + beta (1 - exp(ref_r - logp_r))), the
//            upstream gradient of the backward.
//
// Determinism: one CTA of 1024 threads sums in a fixed order -- thread i
// adds rows i, i + 1024, ... in FP64 (the per-token terms are FP32, the
// inputs' precision), then a fixed shuffle and shared-memory tree -- so the
// loss is bitwise reproducible for a given input whatever the GPU; the count
// N is an exact sum.  The gradient needs N first, so
// the kernel computes both in one CTA: count, then losses, then gradients.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <string>

#include "rlk_internal.h"

namespace rlk {
namespace {

constexpr int kLossThreads = 1024;

__device__ __forceinline__ double block_sum(double v, double* sh) {
#pragma unroll
    for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    double r = 0.0;
    if (warp == 0) {
        r = lane < (kLossThreads / 32) ? sh[lane] : 0.0;
#pragma unroll
        for (int off = 16; off; off >>= 1) r += __shfl_xor_sync(0xFFFFFFFFu, r, off);
    }
    __syncthreads();
    if (threadIdx.x == 0) sh[0] = r;
    __syncthreads();
    r = sh[0];
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kLossThreads, 1)
    grpo_loss_kernel(int64_t T, const float* logp, const float* adv, const uint8_t* mask, const float* ref,
                     float beta, float* loss, float* grad, float* count) {
    __shared__ double sh[kLossThreads / 32];
    double n_local = 0.0;
    for (int64_t r = threadIdx.x; r < T; r += kLossThreads) n_local += (mask[r] != 0) ? 1.0 : 0.0;
    const double n = block_sum(n_local, sh);
    const double inv_n = n > 0.0 ? 1.0 / n : 0.0;
    const float inv_nf = (float)inv_n;
    double acc = 0.0;
    for (int64_t r = threadIdx.x; r < T; r += kLossThreads) {
        // per-token terms in FP32 (the inputs' precision), the sum in FP64
        const bool act = mask[r] != 0;
        const float lp = logp[r], a = adv[r];
        float term = -a * lp, dterm = -a;
        if (ref) {
            const float d = ref[r] - lp;
            const float e = expf(d);
            term = fmaf(beta, (e - d) - 1.f, term);
            dterm = fmaf(beta, 1.f - e, dterm);
        }
        if (act) acc += (double)term;
        grad[r] = act ? dterm * inv_nf : 0.f;
    }
    const double total = block_sum(acc, sh);
    if (threadIdx.x == 0) {
        *loss = (float)(total * inv_n);
        if (count) *count = (float)n;
    }
}

}  // namespace

rlk_status launch_grpo_loss(int64_t T, const float* logp, const float* adv, const uint8_t* mask, const float* ref,
                            float beta, float* loss, float* grad, float* count, cudaStream_t stream) {
    grpo_loss_kernel<<<1, kLossThreads, 0, stream>>>(T, logp, adv, mask, ref, beta, loss, grad, count);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("GRPO loss launch: ") + cudaGetErrorString(e));
    return RLK_OK;
}

}  // namespace rlk
