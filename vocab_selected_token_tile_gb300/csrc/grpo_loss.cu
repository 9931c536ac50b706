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
// Layout: one cluster of 8 CTAs of 1024 threads.  Thread t of CTA k takes
// rows k*1024 + t + j*8192 (j = 0, 1, ...), so every pass is coalesced and
// each thread keeps four rows' loads in flight.  Pass 1 forms each row's FP32
// term and unnormalised gradient, writes the latter to grad, and sums the
// terms in FP64 and the active rows as an integer.  The CTAs then exchange
// their (sum, count) through distributed shared memory; every CTA folds the
// eight partials in rank order, so all agree on N, and pass 2 scales its own
// rows of grad by 1/N.  Each step runs in a fixed order -- a thread's rows in
// index order, a fixed xor butterfly in the warp, warps 0..31 by the same
// butterfly, CTAs 0..7 in rank order -- that does not depend on the GPU or on
// timing, so the loss is bitwise reproducible; N is an exact integer sum.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <string>

#include "rlk_internal.h"
#include "rlk_ptx.cuh"

namespace rlk {
namespace {

constexpr int kLossThreads = 1024;
constexpr int kLossCtas = 8;  // one portable cluster
constexpr int64_t kLossStride = (int64_t)kLossThreads * kLossCtas;
constexpr int kLossUnroll = 4;

struct LossPart {
    double sum;
    unsigned long long count;
};

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    return v;
}

__device__ __forceinline__ unsigned long long warp_sum(unsigned long long v) {
#pragma unroll
    for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    return v;
}

__device__ __forceinline__ double ld_cluster_f64(uint32_t addr) {
    double v;
    asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ unsigned long long ld_cluster_u64(uint32_t addr) {
    unsigned long long v;
    asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
    return v;
}

__global__ void __cluster_dims__(kLossCtas, 1, 1) __launch_bounds__(kLossThreads, 1)
    grpo_loss_kernel(int64_t T, const float* __restrict__ logp, const float* __restrict__ adv,
                     const uint8_t* __restrict__ mask, const float* __restrict__ ref, float beta,
                     float* __restrict__ loss, float* __restrict__ grad, float* __restrict__ count) {
    __shared__ double warp_s[kLossThreads / 32];
    __shared__ unsigned long long warp_n[kLossThreads / 32];
    __shared__ LossPart part;    // this CTA's partial, read by every CTA of the cluster
    __shared__ LossPart folded;  // the cluster's total, for this CTA's threads
    const uint32_t rank = cluster_ctarank();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = (int64_t)rank * kLossThreads + threadIdx.x;

    // pass 1: per-row terms in FP32 (the inputs' precision), sums in FP64
    double acc = 0.0;
    unsigned long long n_act = 0;
    for (int64_t base = t0; base < T; base += kLossUnroll * kLossStride) {
        float lp[kLossUnroll], a[kLossUnroll], rf[kLossUnroll];
        bool act[kLossUnroll];
#pragma unroll
        for (int u = 0; u < kLossUnroll; ++u) {
            const int64_t r = base + u * kLossStride;
            const bool in = r < T;
            act[u] = in && mask[r] != 0;
            lp[u] = in ? logp[r] : 0.f;
            a[u] = in ? adv[r] : 0.f;
            rf[u] = (in && ref) ? ref[r] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kLossUnroll; ++u) {
            const int64_t r = base + u * kLossStride;
            float term = -a[u] * lp[u], dterm = -a[u];
            if (ref) {
                const float d = rf[u] - lp[u];
                const float e = expf(d);
                term = fmaf(beta, (e - d) - 1.f, term);
                dterm = fmaf(beta, 1.f - e, dterm);
            }
            if (act[u]) {
                acc += (double)term;
                ++n_act;
            }
            if (grad && r < T) grad[r] = act[u] ? dterm : 0.f;
        }
    }

    // the CTA's partial, then the cluster's fold in rank order
    acc = warp_sum(acc);
    n_act = warp_sum(n_act);
    if (lane == 0) {
        warp_s[warp] = acc;
        warp_n[warp] = n_act;
    }
    __syncthreads();
    if (warp == 0) {
        const double s = warp_sum(warp_s[lane]);
        const unsigned long long c = warp_sum(warp_n[lane]);
        if (lane == 0) part = LossPart{s, c};
    }
    cluster_sync_all();
    if (threadIdx.x == 0) {
        double total = 0.0;
        unsigned long long n = 0;
        for (int k = 0; k < kLossCtas; ++k) {
            const uint32_t remote = mapa_shared(smem_u32(&part), (uint32_t)k);
            total += ld_cluster_f64(remote);
            n += ld_cluster_u64(remote + 8);
        }
        folded = LossPart{total, n};
    }
    cluster_sync_all();  // no CTA leaves while a peer may still read its partial
    const unsigned long long n = folded.count;
    const double inv_n = n > 0 ? 1.0 / (double)n : 0.0;
    if (rank == 0 && threadIdx.x == 0) {
        *loss = (float)(folded.sum * inv_n);
        if (count) *count = (float)n;
    }

    // pass 2: g_r = (unnormalised gradient) / N on this thread's own rows
    const float inv_nf = (float)inv_n;
    for (int64_t base = t0; grad && base < T; base += kLossUnroll * kLossStride) {
        float v[kLossUnroll];
#pragma unroll
        for (int u = 0; u < kLossUnroll; ++u) {
            const int64_t r = base + u * kLossStride;
            v[u] = r < T ? grad[r] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < kLossUnroll; ++u) {
            const int64_t r = base + u * kLossStride;
            if (r < T) grad[r] = v[u] * inv_nf;
        }
    }
}

// N of the fused GRPO step: the active rows of the contract (explicit mask,
// or target != ignore_index), counted with integer atomics (exact in any
// order).  In ignore_index mode each row's activity is also written to
// mask_out for the loss kernel.
__global__ void __launch_bounds__(256) grpo_count_kernel(int64_t T, const int64_t* __restrict__ targets,
                                                         const uint8_t* __restrict__ mask, int64_t ignore_index,
                                                         uint8_t* __restrict__ mask_out,
                                                         unsigned long long* __restrict__ n_active) {
    unsigned long long n = 0;
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < T; r += (int64_t)gridDim.x * blockDim.x) {
        const bool act = mask ? mask[r] != 0 : targets[r] != ignore_index;
        if (mask_out) mask_out[r] = act ? 1 : 0;
        n += act ? 1 : 0;
    }
    n = warp_sum(n);
    if ((threadIdx.x & 31) == 0 && n) atomicAdd(n_active, n);
}

}  // namespace

rlk_status launch_grpo_count(int64_t T, const int64_t* targets, const uint8_t* mask, int64_t ignore_index,
                             uint8_t* mask_out, unsigned long long* n_active, int sm_count, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(n_active, 0, sizeof(unsigned long long), stream);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("clearing the active count: ") + cudaGetErrorString(e));
    if (T > 0) {
        const int64_t want = (T + 255) / 256;
        const int blocks = (int)(want < 4 * (int64_t)sm_count ? want : 4 * (int64_t)sm_count);
        grpo_count_kernel<<<blocks, 256, 0, stream>>>(T, targets, mask, ignore_index, mask_out, n_active);
        e = cudaGetLastError();
        if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("active count launch: ") + cudaGetErrorString(e));
    }
    return RLK_OK;
}

rlk_status launch_grpo_loss(int64_t T, const float* logp, const float* adv, const uint8_t* mask, const float* ref,
                            float beta, float* loss, float* grad, float* count, cudaStream_t stream) {
    grpo_loss_kernel<<<kLossCtas, kLossThreads, 0, stream>>>(T, logp, adv, mask, ref, beta, loss, grad, count);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("GRPO loss launch: ") + cudaGetErrorString(e));
    return RLK_OK;
}

}  // namespace rlk
