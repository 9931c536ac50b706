// Vocabulary-parallel pieces of the path (sm_103a): what one rank of a real
// tensor-parallel group computes on its column shard, and the fold of the
// partials that the ranks have exchanged.
//
// PR #289 "[WS2][PR4][Logp] feat: add distributed TP/CP logprob drift
// report", PR-1 contract commit: each TP rank holds a tile-aligned shard of
// the padded vocabulary, forms the FP32 (max, sumexp) partials of its tiles,
// the partials travel by all-gather, every rank merges all of them in fixed
// global tile order, and the target logit comes from the rank that owns the
// target's column (owner-rank resolution).  Issue #323 "[WS2][Logprob] H100
// validation and reproduction guide", "Six-Case TP/CP Matrix": TP degrees 1,
// 2, 4, 8 give bitwise-identical logp and LSE.
//
// Shard j of T rows holds columns [j*Vs, (j+1)*Vs), Vs = V_padded / tp, as a
// buffer of its own (row stride >= Vs).  Its partials are those of global
// tiles j*NT/tp .. (j+1)*NT/tp - 1: the streaming forward is run on the shard
// as a vocabulary of its own with every row inactive (so no target is read)
// and its per-tile partials kept.  Because Vs is a multiple of 8, the shard's
// 8-column groups are the global ones shifted by a multiple of 8, so every
// tile's partial is bitwise the one rlk_logp_fwd forms on the whole row.  The
// fold below runs the same fold_tiles on the gathered partials, so logp and
// LSE are bitwise those of rlk_logp_fwd.  The shard backward is the streaming
// backward on the shard, with the LSE given and targets of other shards
// taking no one-hot term.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <string>

#include "rlk_fold.cuh"
#include "rlk_internal.h"

namespace rlk {
namespace {

size_t r256(size_t b) { return (b + 255) / 256 * 256; }

// f32(logit[r, t_r]) where this shard holds column t_r of an active row, else 0.
__global__ void shard_target_kernel(const uint16_t* logits, int64_t stride, const int64_t* targets,
                                    const uint8_t* mask, int mask_mode, int64_t ignore_index, int64_t T, int64_t c0,
                                    int64_t c1, float* xt) {
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < T; r += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = targets[r];
        const bool active = (mask_mode == RLK_MASK_EXPLICIT) ? (mask[r] != 0) : (t != ignore_index);
        float x = 0.f;
        if (active && t >= c0 && t < c1) x = __uint_as_float((uint32_t)logits[r * stride + (t - c0)] << 16);
        xt[r] = x;
    }
}

// The identity partial (-inf, 0) for every tile of a shard with no real column.
__global__ void shard_identity_kernel(float2* partials, int64_t n) {
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        partials[i] = make_float2(-INFINITY, 0.f);
}

// Backward inputs of shard j: the activity of each row as an explicit mask,
// and the target's column within the shard (-1 when another shard holds it).
// An active target outside [0, V_real) is reported as on the whole row.
__global__ void shard_remap_kernel(const int64_t* targets, const uint8_t* mask, int mask_mode, int64_t ignore_index,
                                   int64_t T, int64_t Vr, int64_t c0, int64_t c1, int64_t* local_targets,
                                   uint8_t* local_mask, uint32_t* status) {
    for (int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; r < T; r += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = targets[r];
        const bool active = (mask_mode == RLK_MASK_EXPLICIT) ? (mask[r] != 0) : (t != ignore_index);
        local_mask[r] = active ? 1 : 0;
        local_targets[r] = (active && t >= c0 && t < c1) ? t - c0 : -1;
        if (active && (t < 0 || t >= Vr)) atomicOr(status, kStatusTargetRange);
    }
}

// dlogits of a shard with no real column: every element 0.
__global__ void shard_zero_kernel(uint16_t* d, int64_t stride, int64_t T, int64_t cols) {
    const int64_t n = T * cols;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        d[(i / cols) * stride + i % cols] = 0;
}

// Row `row`'s outcome from its LSE: lane 0 writes LSE and logp and reports
// the device conditions; xt is the target logit (read by lane 0 when needed).
__device__ __forceinline__ void finish_row(int64_t row, float l, int64_t t, bool active, float xt, int64_t Vr,
                                           float* logp, float* lse, uint32_t* status) {
    lse[row] = l;
    if (!active) {
        logp[row] = 0.f;
    } else if (t < 0 || t >= Vr) {
        logp[row] = __int_as_float(0x7FC00000);
        atomicOr(status, kStatusTargetRange);
    } else {
        logp[row] = __fsub_rn(xt, l);
    }
    if (active && !isfinite(l)) atomicOr(status, kStatusNonFinite);
}

// LSE and logp of each row from the gathered partials, one row per thread
// (fold_step / fold_finish: the bits of fold_tiles, without the warp's
// shuffles, which bound a warp-per-row fold of many rows).  gathered
// [tp, T, NT/tp] float2 (shard-major, as an all-gather of every rank's
// [T, NT/tp] partials leaves them), gathered_xt [tp, T]; the target logit is
// taken from the shard that holds the target's column.
__global__ void gathered_fold_kernel(const float2* gathered, const float* gathered_xt, const int64_t* targets,
                                     const uint8_t* mask, int mask_mode, int64_t ignore_index, int64_t T, int64_t Vr,
                                     int64_t Vs, int tp, int ntl, float* logp, float* lse, uint32_t* status) {
    for (int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; row < T; row += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = targets[row];
        const bool active = (mask_mode == RLK_MASK_EXPLICIT) ? (mask[row] != 0) : (t != ignore_index);
        const float xt = (active && t >= 0 && t < Vr) ? gathered_xt[(t / Vs) * T + row] : 0.f;
        float M = -INFINITY, S = 0.f;
        for (int sh = 0; sh < tp; ++sh) {
            const float2* part = gathered + ((int64_t)sh * T + row) * ntl;
            for (int l = 0; l < ntl; ++l) fold_step(M, S, part[l]);
        }
        finish_row(row, fold_finish(M, S), t, active, xt, Vr, logp, lse, status);
    }
}

int grid_for(int64_t n, int threads) {
    int64_t g = (n + threads - 1) / threads;
    if (g > 4096) g = 4096;
    return (int)(g < 1 ? 1 : g);
}

rlk_status launched(const char* what) {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string(what) + " launch: " + cudaGetErrorString(e));
    return RLK_OK;
}

}  // namespace

rlk_logp_contract shard_local_contract(const rlk_logp_contract& c, int32_t shard) {
    const int64_t Vs = c.V_padded / c.virtual_tp;
    const int64_t c0 = (int64_t)shard * Vs;
    int64_t vr = c.V_real - c0;
    if (vr < 0) vr = 0;
    if (vr > Vs) vr = Vs;
    rlk_logp_contract l = c;
    l.V_real = vr;
    l.V_padded = Vs;
    l.num_tiles = c.num_tiles / c.virtual_tp;
    l.virtual_tp = 1;
    l.row_stride = c.row_stride ? c.row_stride : Vs;
    l.mask_mode = RLK_MASK_EXPLICIT;
    l.validate = 0;
    return l;
}

// Workspace after the status word: an explicit mask [T], local logp and LSE
// [T] FP32 (the forward), local targets [T] int64 (the backward).
size_t shard_workspace(const rlk_logp_contract& c) {
    return r256((size_t)c.T) + 2 * r256((size_t)c.T * 4) + r256((size_t)c.T * 8);
}

rlk_status launch_shard_fwd(const rlk_logp_contract& c, int32_t shard, const uint16_t* logits, const int64_t* targets,
                            const uint8_t* mask, float* partials, float* target_logit, void* workspace,
                            uint32_t* status, cudaStream_t stream) {
    const rlk_logp_contract l = shard_local_contract(c, shard);
    const int64_t c0 = (int64_t)shard * l.V_padded;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    uint8_t* none = ws;  // every row inactive: partials only, no target is read
    float* logp_l = reinterpret_cast<float*>(ws + r256((size_t)c.T));
    float* lse_l = reinterpret_cast<float*>(ws + r256((size_t)c.T) + r256((size_t)c.T * 4));
    if (l.V_real == 0) {
        shard_identity_kernel<<<grid_for(c.T * l.num_tiles, 256), 256, 0, stream>>>(
            reinterpret_cast<float2*>(partials), c.T * l.num_tiles);
        rlk_status s = launched("shard identity");
        if (s != RLK_OK) return s;
    } else {
        const cudaError_t e = cudaMemsetAsync(none, 0, (size_t)c.T, stream);
        if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("clearing the shard mask: ") + cudaGetErrorString(e));
        StreamArgs a{};
        a.logits = logits;
        a.targets = targets;
        a.mask = none;
        a.logp = logp_l;
        a.lse = lse_l;
        a.partials = partials;
        a.status = status;
        rlk_status s = launch_stream(l, kModeFwd, a, stream);
        if (s != RLK_OK) return s;
    }
    shard_target_kernel<<<grid_for(c.T, 256), 256, 0, stream>>>(logits, l.row_stride, targets, mask, c.mask_mode,
                                                                c.ignore_index, c.T, c0, c0 + l.V_real, target_logit);
    return launched("shard target logit");
}

rlk_status launch_gathered_fold(const rlk_logp_contract& c, const float* gathered_partials, const float* gathered_xt,
                                const int64_t* targets, const uint8_t* mask, float* logp, float* lse,
                                uint32_t* status, cudaStream_t stream) {
    gathered_fold_kernel<<<grid_for(c.T, 128), 128, 0, stream>>>(
        reinterpret_cast<const float2*>(gathered_partials), gathered_xt, targets, mask, c.mask_mode, c.ignore_index,
        c.T, c.V_real, c.V_padded / c.virtual_tp, c.virtual_tp, c.num_tiles / c.virtual_tp, logp, lse, status);
    return launched("gathered fold");
}

rlk_status launch_shard_bwd(const rlk_logp_contract& c, int32_t shard, const uint16_t* logits, const int64_t* targets,
                            const uint8_t* mask, const float* lse_in, const float* grad, uint16_t* dlogits,
                            void* workspace, uint32_t* status, cudaStream_t stream) {
    const rlk_logp_contract l = shard_local_contract(c, shard);
    const int64_t c0 = (int64_t)shard * l.V_padded;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    uint8_t* lmask = ws;
    int64_t* ltgt = reinterpret_cast<int64_t*>(ws + r256((size_t)c.T) + 2 * r256((size_t)c.T * 4));
    shard_remap_kernel<<<grid_for(c.T, 256), 256, 0, stream>>>(targets, mask, c.mask_mode, c.ignore_index, c.T,
                                                               c.V_real, c0, c0 + l.V_real, ltgt, lmask, status);
    rlk_status s = launched("shard remap");
    if (s != RLK_OK) return s;
    if (l.V_real == 0) {
        shard_zero_kernel<<<grid_for(c.T * l.V_padded, 256), 256, 0, stream>>>(dlogits, l.row_stride, c.T,
                                                                               l.V_padded);
        return launched("shard zero");
    }
    StreamArgs a{};
    a.logits = logits;
    a.dlogits = dlogits;
    a.targets = ltgt;
    a.mask = lmask;
    a.grad = grad;
    a.lse_in = lse_in;
    a.status = status;
    a.foreign_targets = 1;
    return launch_stream(l, kModeBwd, a, stream);
}

}  // namespace rlk
