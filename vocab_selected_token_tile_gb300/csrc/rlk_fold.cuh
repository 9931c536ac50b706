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

// Up to 64 tiles the fold keeps everything in registers: lane l holds tiles
// l and l + 32, the two prefix-max scans run interleaved, and the recurrence
// runs warp-uniformly on values broadcast by shuffles, which do not depend on
// S and so issue ahead of the FMA chain.  Every value is formed by exactly
// the operations of the general path below, in the same order, so both give
// the same bits.
struct FoldTerms {
    float f[2];  // rescale factors f_k = exp(M_{k-1} - M_k) of tiles lane, lane + 32
    float e[2];  // exp(m_k - M_k), 0 for an identity tile
    float b[2];  // terms b_k = s_k exp(m_k - M_k)
    float M;     // the prefix max over all tiles (the row's max)
};

__device__ __forceinline__ FoldTerms fold_terms64(const float2 (&p)[2], int lane) {
    float v0 = p[0].x, v1 = p[1].x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float o0 = __shfl_up_sync(0xFFFFFFFFu, v0, off);
        const float o1 = __shfl_up_sync(0xFFFFFFFFu, v1, off);
        if (lane >= off) {
            v0 = fmax_nan(v0, o0);
            v1 = fmax_nan(v1, o1);
        }
    }
    float M[2];
    M[0] = fmax_nan(-INFINITY, v0);
    const float carry = __shfl_sync(0xFFFFFFFFu, M[0], 31);
    M[1] = fmax_nan(carry, v1);
    float Mp[2] = {__shfl_up_sync(0xFFFFFFFFu, M[0], 1), __shfl_up_sync(0xFFFFFFFFu, M[1], 1)};
    if (lane == 0) {
        Mp[0] = -INFINITY;
        Mp[1] = carry;
    }
    FoldTerms t;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        t.f[h] = (Mp[h] == -INFINITY) ? 0.f : ex2_approx(__fmul_rn(__fsub_rn(Mp[h], M[h]), kLog2e));
        t.e[h] = (p[h].x == -INFINITY) ? 0.f : ex2_approx(__fmul_rn(__fsub_rn(p[h].x, M[h]), kLog2e));
        t.b[h] = (p[h].x == -INFINITY) ? 0.f : __fmul_rn(p[h].y, t.e[h]);
    }
    t.M = __shfl_sync(0xFFFFFFFFu, M[1], 31);
    return t;
}

__device__ __forceinline__ void load_parts64(const float2* part, int NT, int lane, float2 (&p)[2]) {
    p[0] = lane < NT ? part[lane] : make_float2(-INFINITY, 0.f);
    p[1] = lane + 32 < NT ? part[lane + 32] : make_float2(-INFINITY, 0.f);
}

// Left fold of part[0..NT) by one warp; returns LSE = m + log s in every lane
// (-inf when every tile is the identity; NaN propagates).  The running maxima
// M_k are an exact prefix max; the rescale factors f_k = exp(M_{k-1} - M_k)
// and the terms b_k = s_k exp(m_k - M_k) are formed lane-parallel (beyond 64
// tiles into scratch[0..NT)); the sum recurrence S_k = S_{k-1} f_k + b_k then
// runs in index order.
//
// UNROLL: of the 64-step recurrence when NT <= 64 (64: fully unrolled).  The
// steps run in index order either way, so the bits do not depend on it.
template <int UNROLL = 64>
__device__ __forceinline__ float fold_tiles(const float2* part, int NT, float2* scratch, int lane) {
    if (NT <= 64) {
        float2 p[2];
        load_parts64(part, NT, lane, p);
        const FoldTerms t = fold_terms64(p, lane);
        float S = 0.f;
        if constexpr (UNROLL >= 64) {
#pragma unroll
            for (int k = 0; k < 64; ++k) {
                const float f = __shfl_sync(0xFFFFFFFFu, t.f[k >> 5], k & 31);
                const float b = __shfl_sync(0xFFFFFFFFu, t.b[k >> 5], k & 31);
                if (k < NT) S = __fmaf_rn(S, f, b);
            }
        } else {
            // k = 32 h + j; h fixed per half keeps t.f[h] and t.b[h] in registers
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll UNROLL
                for (int j = 0; j < 32; ++j) {
                    const float f = __shfl_sync(0xFFFFFFFFu, t.f[h], j);
                    const float b = __shfl_sync(0xFFFFFFFFu, t.b[h], j);
                    if (32 * h + j < NT) S = __fmaf_rn(S, f, b);
                }
            }
        }
        return (t.M == -INFINITY) ? -INFINITY : __fadd_rn(t.M, logf(S));
    }
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

// The same fold by one thread, one tile at a time, for kernels that fold
// many rows at once (one row per thread): fold_step takes tile k's partial
// in index order, fold_finish gives the LSE.  Every value is formed by the
// operations fold_tiles uses, in the same order -- the running maximum M_k
// is the exact prefix max (max is exact, so the order of a scan does not
// change it), f_k = exp(M_{k-1} - M_k) (0 while M_{k-1} = -inf), the term
// b_k = s_k exp(m_k - M_k) (0 for an identity tile), S = S f_k + b_k -- so
// the bits are those of fold_tiles.
__device__ __forceinline__ void fold_step(float& M, float& S, float2 pk) {
    const float Mk = fmax_nan(M, pk.x);
    const float f = (M == -INFINITY) ? 0.f : ex2_approx(__fmul_rn(__fsub_rn(M, Mk), kLog2e));
    const float b =
        (pk.x == -INFINITY) ? 0.f : __fmul_rn(pk.y, ex2_approx(__fmul_rn(__fsub_rn(pk.x, Mk), kLog2e)));
    S = __fmaf_rn(S, f, b);
    M = Mk;
}

__device__ __forceinline__ float fold_finish(float M, float S) {
    return (M == -INFINITY) ? -INFINITY : __fadd_rn(M, logf(S));
}

// fold_tiles plus the entropy of the row's softmax.  tpart[k] holds the
// tile's t_k = sum_c e^(x_c - m_k) x_c.  The LSE comes from exactly the same
// operations as fold_tiles; beside S the same recurrence runs T_k =
// T_{k-1} f_k + t_k e^(m_k - M_k), so that T / S = sum_c p_c x_c, and the
// entropy -sum_c p_c log p_c = LSE - T / S.  Returns (LSE, entropy) in every
// lane; the entropy is NaN when the LSE is not finite.
__device__ __forceinline__ float2 fold_tiles_ent(const float2* part, const float* tpart, int NT, float2* scratch,
                                                 float* scratch_t, int lane) {
    if (NT <= 64) {
        float2 p[2];
        load_parts64(part, NT, lane, p);
        const FoldTerms t = fold_terms64(p, lane);
        float te[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int k = lane + 32 * h;
            te[h] = (k >= NT || p[h].x == -INFINITY) ? 0.f : __fmul_rn(tpart[k], t.e[h]);
        }
        float S = 0.f, Tt = 0.f;
#pragma unroll
        for (int k = 0; k < 64; ++k) {
            const float f = __shfl_sync(0xFFFFFFFFu, t.f[k >> 5], k & 31);
            const float b = __shfl_sync(0xFFFFFFFFu, t.b[k >> 5], k & 31);
            const float tk = __shfl_sync(0xFFFFFFFFu, te[k >> 5], k & 31);
            if (k < NT) {
                S = __fmaf_rn(S, f, b);
                Tt = __fmaf_rn(Tt, f, tk);
            }
        }
        const float lse = (t.M == -INFINITY) ? -INFINITY : __fadd_rn(t.M, logf(S));
        const float ent = isfinite(lse) ? __fsub_rn(lse, __fdiv_rn(Tt, S)) : __int_as_float(0x7FC00000);
        return make_float2(lse, ent);
    }
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
