// Streaming kernels of the selected-token log-probability path (sm_103a).
//
// One persistent kernel template serves the three streaming entry points:
//
//   kModeFwd   per-tile (max, sumexp) partials -> cluster exchange -> fixed-
//              order fold -> LSE, logp                 (rlk_logp_fwd)
//   kModeBwd   dlogits = g * (onehot - exp(x - LSE)) from a given LSE
//                                                       (rlk_logp_bwd, lse_in)
//   kModeFused both, with each row's slice held in shared memory between the
//              two phases so the logits are read from HBM once
//                                                       (rlk_logp_bwd, no lse_in)
//
// Method (PR #289 "[WS2][PR4][Logp] feat: add distributed TP/CP logprob drift
// report": the PR-1 contract commit, the global-tile commit and the typed
// contract commit): padded columns are -inf; the vocabulary is cut into
// num_tiles global tiles; each tile gives an FP32 (max, sumexp) partial, the
// identity (-inf, 0) when it has no finite column; partials are merged in
// fixed global tile order.  Virtual TP (the H100 matrix document, "Fixes
// exercised": fixed virtual TP8) is a cluster of virtual_tp CTAs: CTA j owns
// the tile-aligned shard j, computes its tiles' partials and pushes them into
// every peer's shared memory (the on-chip analogue of the pages' all-gather);
// every CTA then folds all num_tiles partials in index order, so the result
// does not depend on virtual_tp.
//
// Layout of work.  Cluster q handles rows q, q + G, q + 2G, ... (G clusters).
// Within a CTA, warp kConsumerWarps is the producer: lane 0 streams each
// (row, tile) item's 16-byte-aligned column span into a ring slot with a 1-D
// bulk copy (cp.async.bulk, completion on the slot's "full" mbarrier).  The
// other warps consume items round-robin; one warp reduces one tile.  Within a
// tile the order of arithmetic depends only on the tile's columns: lane l
// takes 8-column groups l, l+32, ... from the aligned start; the exact tile
// maximum is formed first (packed BF16 max), then sum exp(x - m) in FP32, and
// the lanes are combined by a fixed xor butterfly.
//
// Every device-side wait is bounded (wait_timeout_ns): on expiry the kernel
// records RLK_ERR_TIMEOUT in the status word, stops issuing work, drains its
// own bulk copies and returns.  No atomics touch any result; the status word
// is the only atomic target.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <cstdlib>
#include <mutex>
#include <string>

#include "rlk_internal.h"
#include "rlk_ptx.cuh"

namespace rlk {
namespace {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxSlots = 96;
constexpr float kLog2e = 1.4426950408889634f;  // log2(e): e^y = 2^(y log2 e)
constexpr uint64_t kDrainNs = 1000000000ull;   // bound of the final drain of own copies

struct SlotHdr {  // row metadata the producer writes beside each slot
    int64_t target;
    float g;
    float lse_in;
    int32_t active;
    int32_t pad;
    int64_t row;
};
static_assert(sizeof(SlotHdr) == 32, "SlotHdr layout");

struct RowShared {  // per-row state of the fold, double-buffered by row parity
    int64_t target;
    float g;
    int32_t active;
    float xt;       // f32(logit[row, target]) when this CTA owns the target's tile
    int32_t has_xt;
    float lse;
    int32_t pad;
};
static_assert(sizeof(RowShared) == 32, "RowShared layout");

struct Params {
    StreamArgs a;
    int64_t T, Vr, Vp, stride, ignore_index;
    uint64_t wait_ns;
    int32_t NT, W, C, mask_mode, NS, slot_bytes;
    uint32_t off_full, off_empty, off_hdr, off_part, off_fold, off_rows, off_xbar, off_flag;
};

struct TileGeom {
    int64_t ts, te;  // tile columns [ts, te)
    int64_t hi;      // min(te, V_real): end of the tile's real columns
    int64_t a, b;    // slot span [a, b): a = floor8(ts), b = min(ceil8(te), floor8(V_real))
};

__device__ __forceinline__ TileGeom tile_geom(int k, const Params& p) {
    TileGeom t;
    t.ts = (int64_t)k * p.W;
    t.te = t.ts + p.W;
    t.hi = t.te < p.Vr ? t.te : p.Vr;
    t.a = t.ts & ~(int64_t)7;
    const int64_t ce = (t.te + 7) & ~(int64_t)7;
    const int64_t fv = p.Vr & ~(int64_t)7;
    t.b = ce < fv ? ce : fv;
    return t;
}

// ----------------------------------------------------------------- bounded waits

struct Waiter {
    volatile int* abort_flag;
    uint32_t* status;
    uint64_t limit_ns;

    __device__ bool wait(uint32_t bar, uint32_t parity, bool cluster_scope) const {
        auto poll = [&]() { return cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
        if (poll()) return true;
        if (*abort_flag) return false;
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
            if (poll()) return true;
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                *abort_flag = 1;
                atomicOr(status, kStatusTimeout);
                return false;
            }
        }
    }
    // All 32 lanes wait (each acquires the barrier's phase); the warp agrees on the outcome.
    __device__ bool warp_wait(uint32_t bar, uint32_t parity, bool cluster_scope = false) const {
        const bool ok = wait(bar, parity, cluster_scope);
        const bool all = __all_sync(0xFFFFFFFFu, ok);
        if (!all) *abort_flag = 1;
        return all;
    }
};

// ----------------------------------------------------------------- per-tile work

__device__ __forceinline__ uint32_t neg_inf_lo(uint32_t w) { return (w & 0xFFFF0000u) | 0xFF80u; }
__device__ __forceinline__ uint32_t neg_inf_hi(uint32_t w) { return (w & 0x0000FFFFu) | 0xFF800000u; }

__device__ __forceinline__ uint16_t ldg_bf16(const uint16_t* p) {
    return __ldg(reinterpret_cast<const unsigned short*>(p));
}

// The 8 BF16 values of columns [c0, c0+8) as a uint4; columns outside the
// tile's real range [ts, hi) read as -inf.  Groups inside the slot span come
// from shared memory; the ragged real tail [floor8(V_real), V_real) is read
// from global memory one element at a time.
__device__ __forceinline__ uint4 load_group(const uint16_t* slot, const uint16_t* grow, int64_t c0,
                                            const TileGeom& t) {
    uint4 v;
    if (c0 + 8 <= t.b) {
        v = *reinterpret_cast<const uint4*>(slot + (c0 - t.a));
    } else {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t c = c0 + 2 * j;
            const uint32_t lo = (c < t.hi && c >= t.ts) ? ldg_bf16(grow + c) : 0xFF80u;
            const uint32_t hi = (c + 1 < t.hi && c + 1 >= t.ts) ? ldg_bf16(grow + c + 1) : 0xFF80u;
            w[j] = lo | (hi << 16);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (c0 < t.ts || c0 + 8 > t.hi) {
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t c = c0 + 2 * j;
            if (c < t.ts || c >= t.hi) w[j] = neg_inf_lo(w[j]);
            if (c + 1 < t.ts || c + 1 >= t.hi) w[j] = neg_inf_hi(w[j]);
        }
        v = make_uint4(w[0], w[1], w[2], w[3]);
    }
    return v;
}

__device__ __forceinline__ float warp_max_nan(float v) {
#pragma unroll
    for (int off = 16; off; off >>= 1) v = fmax_nan(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int off = 16; off; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
    return v;
}

__device__ __forceinline__ float exp_term(float x, float neg_mL) {
    return ex2_approx(__fmaf_rn(x, kLog2e, neg_mL));
}

// (m_k, s_k) of one tile, computed by one warp; every lane returns the same value.
__device__ float2 tile_partial(const uint16_t* slot, const uint16_t* grow, const TileGeom& t, int lane) {
    if (t.hi <= t.ts) return make_float2(-INFINITY, 0.f);  // padding-only tile: identity
    const int ng = (int)((((t.hi + 7) & ~(int64_t)7) - t.a) >> 3);
    uint32_t acc0 = 0xFF80FF80u, acc1 = 0xFF80FF80u;
#pragma unroll 4
    for (int gi = lane; gi < ng; gi += 32) {
        const uint4 v = load_group(slot, grow, t.a + 8 * (int64_t)gi, t);
        acc0 = bf16x2_max_nan(acc0, v.x);
        acc1 = bf16x2_max_nan(acc1, v.y);
        acc0 = bf16x2_max_nan(acc0, v.z);
        acc1 = bf16x2_max_nan(acc1, v.w);
    }
    acc0 = bf16x2_max_nan(acc0, acc1);
    const float m = warp_max_nan(fmax_nan(bf16lo_to_f32(acc0), bf16hi_to_f32(acc0)));
    if (m == -INFINITY) return make_float2(-INFINITY, 0.f);  // all -inf: identity
    const float nmL = -__fmul_rn(m, kLog2e);
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll 4
    for (int gi = lane; gi < ng; gi += 32) {
        const uint4 v = load_group(slot, grow, t.a + 8 * (int64_t)gi, t);
        s0 = __fadd_rn(s0, exp_term(bf16lo_to_f32(v.x), nmL));
        s1 = __fadd_rn(s1, exp_term(bf16hi_to_f32(v.x), nmL));
        s2 = __fadd_rn(s2, exp_term(bf16lo_to_f32(v.y), nmL));
        s3 = __fadd_rn(s3, exp_term(bf16hi_to_f32(v.y), nmL));
        s0 = __fadd_rn(s0, exp_term(bf16lo_to_f32(v.z), nmL));
        s1 = __fadd_rn(s1, exp_term(bf16hi_to_f32(v.z), nmL));
        s2 = __fadd_rn(s2, exp_term(bf16lo_to_f32(v.w), nmL));
        s3 = __fadd_rn(s3, exp_term(bf16hi_to_f32(v.w), nmL));
    }
    const float s = warp_sum(__fadd_rn(__fadd_rn(s0, s1), __fadd_rn(s2, s3)));
    return make_float2(m, s);
}

// dlogits of one tile's columns [ts, te) of one row, by one warp.
__device__ void tile_grad(const uint16_t* slot, const uint16_t* grow, uint16_t* drow, const TileGeom& t,
                          int64_t Vr, bool active, int64_t target, float g, float lse, int lane) {
    const int64_t ce = (t.te + 7) & ~(int64_t)7;
    const int ng = (int)((ce - t.a) >> 3);
    if (!active) {
        for (int gi = lane; gi < ng; gi += 32) {
            const int64_t c0 = t.a + 8 * (int64_t)gi;
            if (c0 >= t.ts && c0 + 8 <= t.te) {
                __stcs(reinterpret_cast<uint4*>(drow + c0), make_uint4(0u, 0u, 0u, 0u));
            } else {
                for (int e = 0; e < 8; ++e) {
                    const int64_t c = c0 + e;
                    if (c >= t.ts && c < t.te) drow[c] = 0;
                }
            }
        }
        return;
    }
    const float nlL = -__fmul_rn(lse, kLog2e);
    const float ng_ = -g;
    const bool tgt_ok = target >= 0 && target < Vr;
#pragma unroll 2
    for (int gi = lane; gi < ng; gi += 32) {
        const int64_t c0 = t.a + 8 * (int64_t)gi;
        float pr[8];
        bool fast = c0 + 8 <= t.b;
        if (fast) {
            const uint4 v = *reinterpret_cast<const uint4*>(slot + (c0 - t.a));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                pr[2 * j] = exp_term(bf16lo_to_f32(w[j]), nlL);
                pr[2 * j + 1] = exp_term(bf16hi_to_f32(w[j]), nlL);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int64_t c = c0 + e;
                pr[e] = (c < Vr) ? exp_term(__uint_as_float((uint32_t)ldg_bf16(grow + c) << 16), nlL) : 0.f;
            }
        }
        float d[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) d[e] = __fmul_rn(ng_, pr[e]);
        if (!fast) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (c0 + e >= Vr) d[e] = 0.f;  // padded column: exactly +0
        }
        if (tgt_ok && (uint64_t)(target - c0) < 8u) {
            const int e = (int)(target - c0);
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j == e) d[j] = __fmul_rn(g, __fsub_rn(1.f, pr[j]));
        }
        const uint32_t w0 = pack_bf16x2_rn(d[0], d[1]), w1 = pack_bf16x2_rn(d[2], d[3]);
        const uint32_t w2 = pack_bf16x2_rn(d[4], d[5]), w3 = pack_bf16x2_rn(d[6], d[7]);
        if (c0 >= t.ts && c0 + 8 <= t.te) {
            __stcs(reinterpret_cast<uint4*>(drow + c0), make_uint4(w0, w1, w2, w3));
        } else {
            const uint32_t w[4] = {w0, w1, w2, w3};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int64_t c = c0 + e;
                if (c >= t.ts && c < t.te) drow[c] = (uint16_t)((e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xFFFFu));
            }
        }
    }
}

// ----------------------------------------------------------------- kernel roles

struct Ctx {
    int warp, lane;
    uint32_t rank;
    int64_t q, G, nrows;
    int k0, ntl;
    unsigned char* smem;
    uint32_t sbase, full0, empty0, xbar0;
    SlotHdr* hdr;
    float2* part;
    float2* fold;
    RowShared* rows;
    Waiter wt;
};

template <int MODE>
__device__ void producer(const Params& p, const Ctx& x) {
    const int lane = x.lane;
    const uint64_t policy = l2_policy_evict_first();
    int64_t meta_base = 0;
    int64_t m_t = 0;
    int32_t m_act = 0;
    float m_g = 0.f, m_l = 0.f;
    auto load_meta = [&](int64_t base) {
        const int64_t n = base + lane;
        if (n < x.nrows) {
            const int64_t r = x.q + n * x.G;
            m_t = p.a.targets[r];
            m_act = (p.mask_mode == RLK_MASK_EXPLICIT) ? (p.a.mask[r] != 0) : (m_t != p.ignore_index);
            m_g = (MODE != kModeFwd) ? p.a.grad[r] : 0.f;
            m_l = (MODE == kModeBwd) ? p.a.lse_in[r] : 0.f;
        }
    };
    load_meta(0);
    int64_t issued = 0;
    int slot = 0;
    uint32_t phase = 0;
    bool aborted = false;
    for (int64_t n = 0; n < x.nrows && !aborted; ++n) {
        if (n - meta_base >= 32) {
            meta_base = n;
            load_meta(n);
        }
        const int src = (int)(n - meta_base);
        const int64_t t = (int64_t)__shfl_sync(0xFFFFFFFFu, (unsigned long long)m_t, src);
        const int32_t act = __shfl_sync(0xFFFFFFFFu, m_act, src);
        const float g = __shfl_sync(0xFFFFFFFFu, m_g, src);
        const float lin = __shfl_sync(0xFFFFFFFFu, m_l, src);
        const int64_t row = x.q + n * x.G;
        const uint16_t* grow = p.a.logits + row * p.stride;
        for (int l = 0; l < x.ntl; ++l) {
            bool ok = true;
            if (lane == 0) ok = x.wt.wait(x.empty0 + 8u * slot, phase ^ 1u, false);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) {
                aborted = true;
                break;
            }
            if (lane == 0) {
                SlotHdr h;
                h.target = t;
                h.g = g;
                h.lse_in = lin;
                h.active = act;
                h.pad = 0;
                h.row = row;
                x.hdr[slot] = h;
                const TileGeom tg = tile_geom(x.k0 + l, p);
                const uint32_t bytes =
                    (tg.b > tg.a && (MODE != kModeBwd || act)) ? (uint32_t)((tg.b - tg.a) * 2) : 0u;
                const uint32_t fb = x.full0 + 8u * slot;
                if (bytes) {
                    mbar_arrive_expect_tx(fb, bytes);
                    bulk_g2s(x.sbase + (uint32_t)slot * (uint32_t)p.slot_bytes, grow + tg.a, bytes, fb, policy);
                } else {
                    mbar_arrive(fb);
                }
            }
            ++issued;
            if (++slot == p.NS) {
                slot = 0;
                phase ^= 1u;
            }
        }
    }
    // Drain: wait (bounded) until every copy this CTA issued has landed.
    if (lane == 0) {
        const int64_t first = issued > p.NS ? issued - p.NS : 0;
        for (int64_t j = first; j < issued; ++j) {
            const uint32_t s = (uint32_t)(j % p.NS), par = (uint32_t)((j / p.NS) & 1);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(x.full0 + 8u * s, par)) {
                if (globaltimer_ns() - t0 > kDrainNs) {
                    atomicOr(p.a.status, kStatusTimeout);
                    break;
                }
            }
        }
    }
}

// Exchange (cluster), fold, outputs: warp 0 of every CTA, after the row's
// partials of this CTA are in part[buf].
template <int MODE>
__device__ void fold_row(const Params& p, const Ctx& x, int64_t n) {
    const int lane = x.lane;
    const int buf = (int)(n & 1);
    float2* part = x.part + (size_t)buf * p.NT;
    bool ok = !*x.wt.abort_flag;
    if (p.C > 1) {
        if (ok && lane < p.C && (uint32_t)lane != x.rank) {
            // Push this CTA's shard of partials into peer `lane`, then release them.
            for (int kk = x.k0; kk < x.k0 + x.ntl; ++kk) {
                const float2 v = part[kk];
                st_cluster_f32x2(mapa_shared(smem_u32(&part[kk]), (uint32_t)lane), v.x, v.y);
            }
            mbar_arrive_remote(mapa_shared(x.xbar0 + 8u * buf, (uint32_t)lane));
        }
        __syncwarp();
        ok = x.wt.warp_wait(x.xbar0 + 8u * buf, (uint32_t)((n >> 1) & 1), true) && ok;
    }
    if (!ok) return;
    // Left fold over k = 0..NT-1.  The running maxima M_k are an exact prefix
    // max; the rescale factors f_k = exp(M_{k-1} - M_k) and the terms
    // b_k = s_k exp(m_k - M_k) are formed lane-parallel; the sum recurrence
    // S_k = S_{k-1} f_k + b_k then runs in index order in one lane.
    float carry = -INFINITY;
    for (int c0 = 0; c0 < p.NT; c0 += 32) {
        const int k = c0 + lane;
        const float2 pk = k < p.NT ? part[k] : make_float2(-INFINITY, 0.f);
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
        const float b = (pk.x == -INFINITY) ? 0.f : __fmul_rn(pk.y, ex2_approx(__fmul_rn(__fsub_rn(pk.x, Mk), kLog2e)));
        if (k < p.NT) x.fold[k] = make_float2(f, b);
        carry = __shfl_sync(0xFFFFFFFFu, Mk, 31);
    }
    __syncwarp();
    float lse_v = 0.f;
    if (lane == 0) {
        float S = 0.f;
        for (int k = 0; k < p.NT; ++k) {
            const float2 fb = x.fold[k];
            S = __fmaf_rn(S, fb.x, fb.y);
        }
        lse_v = (carry == -INFINITY) ? -INFINITY : __fadd_rn(carry, logf(S));
    }
    lse_v = __shfl_sync(0xFFFFFFFFu, lse_v, 0);
    const int64_t row = x.q + n * x.G;
    if (lane == 0) {
        RowShared& rs = x.rows[buf];
        const bool active = rs.active != 0;
        const int64_t t = rs.target;
        if (x.rank == 0) {
            p.a.lse[row] = lse_v;
            if (!active) {
                p.a.logp[row] = 0.f;
            } else if (t < 0 || t >= p.Vr) {
                p.a.logp[row] = __int_as_float(0x7FC00000);
                atomicOr(p.a.status, kStatusTargetRange);
            }
            if (active && !isfinite(lse_v)) atomicOr(p.a.status, kStatusNonFinite);
        }
        if (active && rs.has_xt) p.a.logp[row] = __fsub_rn(rs.xt, lse_v);
        rs.has_xt = 0;
        rs.lse = lse_v;
    }
    if (p.a.partials && x.rank == 0) {
        float2* out = reinterpret_cast<float2*>(p.a.partials) + row * p.NT;
        for (int k = lane; k < p.NT; k += 32) out[k] = part[k];
    }
}

template <int MODE>
__device__ void consumer(const Params& p, const Ctx& x) {
    const int W = kConsumerWarps;
    const int lane = x.lane;
    uint16_t* slots = reinterpret_cast<uint16_t*>(x.smem);
    const int slot_elems = p.slot_bytes / 2;
    if constexpr (MODE == kModeBwd) {
        const int64_t total = x.nrows * x.ntl;
        for (int64_t i = x.warp; i < total; i += W) {
            const int slot = (int)(i % p.NS);
            if (!x.wt.warp_wait(x.full0 + 8u * slot, (uint32_t)((i / p.NS) & 1))) continue;
            const SlotHdr h = x.hdr[slot];
            const int k = (int)(i % x.ntl);
            const TileGeom tg = tile_geom(x.k0 + k, p);
            if (k == 0 && lane == 0 && h.active) {
                if (h.target < 0 || h.target >= p.Vr) atomicOr(p.a.status, kStatusTargetRange);
                if (!isfinite(h.lse_in)) atomicOr(p.a.status, kStatusNonFinite);
            }
            tile_grad(slots + (size_t)slot * slot_elems, p.a.logits + h.row * p.stride,
                      p.a.dlogits + h.row * p.stride, tg, p.Vr, h.active != 0, h.target, h.g, h.lse_in, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(x.empty0 + 8u * slot);
        }
    } else {
    for (int64_t n = 0; n < x.nrows; ++n) {
        const int buf = (int)(n & 1);
        const int64_t ibase = n * x.ntl;
        const int lfirst = (int)((x.warp - (int)(ibase % W) + W) % W);
        bool row_ok = true;  // every phase-A wait of this warp in this row succeeded
        for (int l = lfirst; l < x.ntl; l += W) {
            const int64_t i = ibase + l;
            const int slot = (int)(i % p.NS);
            if (!x.wt.warp_wait(x.full0 + 8u * slot, (uint32_t)((i / p.NS) & 1))) {
                row_ok = false;
                continue;
            }
            const SlotHdr h = x.hdr[slot];
            const TileGeom tg = tile_geom(x.k0 + l, p);
            const uint16_t* sl = slots + (size_t)slot * slot_elems;
            const uint16_t* grow = p.a.logits + h.row * p.stride;
            const float2 pr = tile_partial(sl, grow, tg, lane);
            if (lane == 0) {
                x.part[(size_t)buf * p.NT + x.k0 + l] = pr;
                RowShared& rs = x.rows[buf];
                if (l == 0) {
                    rs.target = h.target;
                    rs.active = h.active;
                    rs.g = h.g;
                }
                if (h.active && h.target >= tg.ts && h.target < tg.hi) {
                    const uint16_t bits = (h.target < tg.b) ? sl[h.target - tg.a] : ldg_bf16(grow + h.target);
                    rs.xt = __uint_as_float((uint32_t)bits << 16);
                    rs.has_xt = 1;
                }
            }
            if (MODE == kModeFwd) {
                __syncwarp();
                if (lane == 0) mbar_arrive(x.empty0 + 8u * slot);
            }
        }
        named_bar_sync(1, W * 32);
        if (x.warp == 0) fold_row<MODE>(p, x, n);
        if (MODE == kModeFused) {
            named_bar_sync(2, W * 32);
            // After an expired wait the slot headers may be stale: skip the
            // writes (the status word already says RLK_ERR_TIMEOUT).
            if (!row_ok || *x.wt.abort_flag) continue;
            const float lse_v = x.rows[buf].lse;
            for (int l = lfirst; l < x.ntl; l += W) {
                const int64_t i = ibase + l;
                const int slot = (int)(i % p.NS);
                const SlotHdr h = x.hdr[slot];
                const TileGeom tg = tile_geom(x.k0 + l, p);
                tile_grad(slots + (size_t)slot * slot_elems, p.a.logits + h.row * p.stride,
                          p.a.dlogits + h.row * p.stride, tg, p.Vr, h.active != 0, h.target, h.g, lse_v, lane);
                __syncwarp();
                if (lane == 0) mbar_arrive(x.empty0 + 8u * slot);
            }
        }
    }
    }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) stream_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) unsigned char smem[];
    Ctx x;
    x.warp = threadIdx.x >> 5;
    x.lane = threadIdx.x & 31;
    x.rank = (p.C > 1) ? cluster_ctarank() : 0u;
    x.q = blockIdx.x / p.C;
    x.G = gridDim.x / p.C;
    x.nrows = (x.q < p.T) ? (p.T - 1 - x.q) / x.G + 1 : 0;
    x.k0 = (int)(((int64_t)x.rank * p.NT) / p.C);
    x.ntl = (int)(((int64_t)(x.rank + 1) * p.NT) / p.C) - x.k0;
    x.smem = smem;
    x.sbase = smem_u32(smem);
    x.full0 = x.sbase + p.off_full;
    x.empty0 = x.sbase + p.off_empty;
    x.xbar0 = x.sbase + p.off_xbar;
    x.hdr = reinterpret_cast<SlotHdr*>(smem + p.off_hdr);
    x.part = reinterpret_cast<float2*>(smem + p.off_part);
    x.fold = reinterpret_cast<float2*>(smem + p.off_fold);
    x.rows = reinterpret_cast<RowShared*>(smem + p.off_rows);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.off_flag);
    x.wt.abort_flag = abort_flag;
    x.wt.status = p.a.status;
    x.wt.limit_ns = p.wait_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.NS; ++s) {
            mbar_init(x.full0 + 8u * s, 1);
            mbar_init(x.empty0 + 8u * s, 1);
        }
        if (p.C > 1) {
            mbar_init(x.xbar0, (uint32_t)(p.C - 1));
            mbar_init(x.xbar0 + 8u, (uint32_t)(p.C - 1));
        }
        *abort_flag = 0;
        x.rows[0].has_xt = 0;
        x.rows[1].has_xt = 0;
        fence_mbar_init();
    }
    if (p.C > 1) cluster_sync_all(); else __syncthreads();

    if (x.warp == kConsumerWarps) producer<MODE>(p, x);
    else consumer<MODE>(p, x);

    __syncthreads();
    if (p.C > 1) cluster_sync_all();  // no CTA leaves while a peer may still write into it
}

// ----------------------------------------------------------------- host planning

struct DeviceInfo {
    int sm_count = 0;
    int smem_optin = 0;
};

DeviceInfo device_info(int dev) {
    static std::mutex mu;
    static DeviceInfo cache[64];
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && cache[dev].sm_count) return cache[dev];
    DeviceInfo d;
    cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (dev >= 0 && dev < 64) cache[dev] = d;
    return d;
}

int env_int(const char* name, int dflt) {
    const char* v = std::getenv(name);
    return (v && *v) ? std::atoi(v) : dflt;
}

uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Shared-memory layout for NS slots; returns the total bytes.
uint32_t layout(Params& p, int NS) {
    uint32_t off = (uint32_t)NS * (uint32_t)p.slot_bytes;
    p.off_full = off;
    off += 8u * NS;
    p.off_empty = off;
    off += 8u * NS;
    p.off_hdr = align_up(off, 16);
    off = p.off_hdr + (uint32_t)sizeof(SlotHdr) * NS;
    p.off_part = align_up(off, 16);
    off = p.off_part + 2u * 8u * (uint32_t)p.NT;
    p.off_fold = off;
    off += 8u * (uint32_t)p.NT;
    p.off_rows = align_up(off, 16);
    off = p.off_rows + 2u * (uint32_t)sizeof(RowShared);
    p.off_xbar = align_up(off, 8);
    off = p.off_xbar + 16u;
    p.off_flag = off;
    off += 16u;
    return align_up(off, 128);
}

}  // namespace

rlk_status launch_stream(const rlk_logp_contract& c, int mode, const StreamArgs& a, cudaStream_t stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(RLK_ERR_CUDA, "cudaGetDevice failed");
    const DeviceInfo di = device_info(dev);
    if (di.sm_count <= 0) return fail(RLK_ERR_CUDA, "cannot query the device");

    Params p{};
    p.a = a;
    p.T = c.T;
    p.Vr = c.V_real;
    p.Vp = c.V_padded;
    p.stride = c.row_stride ? c.row_stride : c.V_padded;
    p.ignore_index = c.ignore_index;
    p.wait_ns = c.wait_timeout_ns > 0 ? (uint64_t)c.wait_timeout_ns : kDefaultWaitNs;
    p.NT = c.num_tiles;
    p.W = (int32_t)(c.V_padded / c.num_tiles);
    p.mask_mode = c.mask_mode;
    p.slot_bytes = (int32_t)align_up((uint32_t)((((p.W + 7) & ~7) + 8) * 2), 16);

    const int ctas_per_sm = env_int("RLK_CTAS_PER_SM", 1) >= 2 ? 2 : 1;
    const uint32_t budget = (uint32_t)di.smem_optin / (uint32_t)ctas_per_sm - 1024u;
    const int cap = env_int("RLK_MAX_SLOTS", kMaxSlots);
    auto max_slots = [&](Params& q) {
        int lo = 0;
        for (int ns = 1; ns <= cap; ++ns) {
            if (layout(q, ns) <= budget) lo = ns;
            else break;
        }
        return lo;
    };

    int C = (mode == kModeBwd) ? 1 : c.virtual_tp;
    int NS = 0;
    p.C = C;
    if (mode == kModeFused) {
        for (;;) {
            p.C = C;
            NS = max_slots(p);
            const int ntl_max = (c.num_tiles + C - 1) / C;
            if (NS >= ntl_max) break;
            C *= 2;
            if (C > 8 || C > c.num_tiles)
                return fail(RLK_ERR_UNSUPPORTED,
                            "vocabulary too large to keep a row's shard resident for the single-pass fused "
                            "forward+backward; call rlk_logp_fwd then rlk_logp_bwd with lse_in");
        }
    } else {
        NS = max_slots(p);
    }
    if (NS < 1) return fail(RLK_ERR_UNSUPPORTED, "tile too wide for one shared-memory slot");
    p.NS = NS;
    const uint32_t smem = layout(p, NS);

    void (*kfn)(Params) = (mode == kModeFwd) ? stream_kernel<kModeFwd>
                        : (mode == kModeBwd) ? stream_kernel<kModeBwd>
                                             : stream_kernel<kModeFused>;
    const void* fn = reinterpret_cast<const void*>(kfn);
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));

    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.numAttrs = 0;
    int64_t clusters = 0;
    if (p.C > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)p.C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3((unsigned)(p.C * (di.sm_count / p.C)), 1, 1);
        int n = 0;
        e = cudaOccupancyMaxActiveClusters(&n, kfn, &cfg);
        if (e != cudaSuccess || n <= 0)
            return fail(RLK_ERR_CUDA, std::string("no cluster of ") + std::to_string(p.C) +
                                          " CTAs fits: " + cudaGetErrorString(e));
        clusters = n;
    } else {
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, smem);
        if (e != cudaSuccess || per_sm <= 0)
            return fail(RLK_ERR_CUDA, std::string("kernel does not fit on an SM: ") + cudaGetErrorString(e));
        clusters = (int64_t)per_sm * di.sm_count;
    }
    if (clusters > p.T) clusters = p.T;
    cfg.gridDim = dim3((unsigned)(clusters * p.C), 1, 1);
    e = cudaLaunchKernelEx(&cfg, kfn, p);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(e));
    return RLK_OK;
}

}  // namespace rlk
