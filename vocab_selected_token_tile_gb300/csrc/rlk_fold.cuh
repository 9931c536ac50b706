// The fixed-order merge of per-tile (max, sumexp) partials, shared by every
// kernel that produces partials, so that all of them fold in exactly the
// same arithmetic.
//
// PR #289 "[WS2][PR4][Logp] feat: add distributed TP/CP logprob drift
// report", PR-1 contract commit: an FP32 (max, sumexp) merge in fixed global
// index order; "typed contract" commit: the (-inf, 0) identity partial.
// Merging (m1, s1) and (m2, s2) gives m = max(m1, m2),
// s = s1 exp(m1 - m) + s2 exp(m2 - m); an operand with m = -inf adds 0.
#pragma once

#include <math.h>
#include <stdint.h>

#include "rlk_ptx.cuh"

namespace rlk {

constexpr float kLog2e = 1.4426950408889634f;  // log2(e): e^y = 2^(y log2 e)

// Left fold of part[0..NT) by one warp; returns LSE = m + log s in every lane
// (-inf when every tile is the identity; NaN propagates).  The running maxima
// M_k are an exact prefix max; the rescale factors f_k = exp(M_{k-1} - M_k)
// and the terms b_k = s_k exp(m_k - M_k) are formed lane-parallel into
// scratch[0..NT); the sum recurrence S_k = S_{k-1} f_k + b_k then runs in
// index order in lane 0.
__device__ __forceinline__ float fold_tiles(const float2* part, int NT, float2* scratch, int lane) {
    float carry = -INFINITY;
    for (int c0 = 0; c0 < NT; c0 += 32) {
        const int k = c0 + lane;
        const float2 pk = k < NT ? part[k] : make_float2(-INFINITY, 0.f);
        float v = pk.x;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(0xFFFFFFFFu, v, off);
            if (lane >= off) v = fmax_nan(v, o);
        }
        const float Mk = fmax_nan(carry, v);
        float Mp = __shfl_up_sync(0xFFFFFFFFu, Mk, 1);
        if (lane == 0) Mp = carry;
        const float f = (Mp == -INFINITY) ? 0.f : ex2_approx(__fmul_rn(__fsub_rn(Mp, Mk), kLog2e));
        const float bk =
            (pk.x == -INFINITY) ? 0.f : __fmul_rn(pk.y, ex2_approx(__fmul_rn(__fsub_rn(pk.x, Mk), kLog2e)));
        if (k < NT) scratch[k] = make_float2(f, bk);
        carry = __shfl_sync(0xFFFFFFFFu, Mk, 31);
    }
    __syncwarp();
    float lse = 0.f;
    if (lane == 0) {
        float S = 0.f;
#pragma unroll 8
        for (int k = 0; k < NT; ++k) {
            const float2 fb = scratch[k];
            S = __fmaf_rn(S, fb.x, fb.y);
        }
        lse = (carry == -INFINITY) ? -INFINITY : __fadd_rn(carry, logf(S));
    }
    return __shfl_sync(0xFFFFFFFFu, lse, 0);
}

// fold_tiles plus the entropy of the row's softmax.  tpart[k] holds the
// tile's t_k = sum_c e^(x_c - m_k) x_c.  The LSE comes from exactly the same
// operations as fold_tiles; beside S the same recurrence runs T_k =
// T_{k-1} f_k + t_k e^(m_k - M_k), so that T / S = sum_c p_c x_c, and the
// entropy -sum_c p_c log p_c = LSE - T / S.  Returns (LSE, entropy) in every
// lane; the entropy is NaN when the LSE is not finite.
__device__ __forceinline__ float2 fold_tiles_ent(const float2* part, const float* tpart, int NT, float2* scratch,
                                                 float* scratch_t, int lane) {
    float carry = -INFINITY;
    for (int c0 = 0; c0 < NT; c0 += 32) {
        const int k = c0 + lane;
        const float2 pk = k < NT ? part[k] : make_float2(-INFINITY, 0.f);
        const float tk = k < NT ? tpart[k] : 0.f;
        float v = pk.x;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float o = __shfl_up_sync(0xFFFFFFFFu, v, off);
            if (lane >= off) v = fmax_nan(v, o);
        }
        const float Mk = fmax_nan(carry, v);
        float Mp = __shfl_up_sync(0xFFFFFFFFu, Mk, 1);
        if (lane == 0) Mp = carry;
        const float f = (Mp == -INFINITY) ? 0.f : ex2_approx(__fmul_rn(__fsub_rn(Mp, Mk), kLog2e));
        const float e = (pk.x == -INFINITY) ? 0.f : ex2_approx(__fmul_rn(__fsub_rn(pk.x, Mk), kLog2e));
        const float bk = (pk.x == -INFINITY) ? 0.f : __fmul_rn(pk.y, e);
        if (k < NT) {
            scratch[k] = make_float2(f, bk);
            scratch_t[k] = (pk.x == -INFINITY) ? 0.f : __fmul_rn(tk, e);
        }
        carry = __shfl_sync(0xFFFFFFFFu, Mk, 31);
    }
    __syncwarp();
    float lse = 0.f, ent = 0.f;
    if (lane == 0) {
        float S = 0.f, Tt = 0.f;
#pragma unroll 8
        for (int k = 0; k < NT; ++k) {
            const float2 fb = scratch[k];
            S = __fmaf_rn(S, fb.x, fb.y);
            Tt = __fmaf_rn(Tt, fb.x, scratch_t[k]);
        }
        lse = (carry == -INFINITY) ? -INFINITY : __fadd_rn(carry, logf(S));
        ent = isfinite(lse) ? __fsub_rn(lse, __fdiv_rn(Tt, S)) : __int_as_float(0x7FC00000);
    }
    return make_float2(__shfl_sync(0xFFFFFFFFu, lse, 0), __shfl_sync(0xFFFFFFFFu, ent, 0));
}

}  // namespace rlk
