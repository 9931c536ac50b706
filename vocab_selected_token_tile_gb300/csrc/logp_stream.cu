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
//   kModeFusedL2 both, streaming like kModeFwd: phase A releases each slot at
//              once and phase B copies the row again, which the L2 still holds
//              (phase-A copies of rows that need a gradient carry an
//              evict-last hint, every other copy evict-first), so HBM still
//              sees one read of the logits; the default for rlk_logp_bwd
//              without lse_in (RLK_FUSED_SCHEDULE=resident selects kModeFused)
//
// Template flags add variants without putting their code in the others: the
// entropy of each row's softmax (kFlagEnt: rlk_logp_fwd_entropy,
// rlk_logp_fwd_bwd_entropy) and the GRPO step's on-chip g (kFlagGrpo:
// rlk_grpo_fused_step).
//
// Method (PR #289 "[WS2][PR4][Logp] feat: add distributed TP/CP logprob drift
// report": the PR-1 contract commit, the global-tile commit and the typed
// contract commit): padded columns are -inf; the vocabulary is cut into
// num_tiles global tiles; each tile gives an FP32 (max, sumexp) partial, the
// identity (-inf, 0) when it has no finite column; partials are merged in
// fixed global tile order.  Virtual TP (the H100 matrix document, "Fixes
// exercised": fixed virtual TP8) is a cluster of virtual_tp CTAs (two at
// virtual TP 1 in kModeFusedL2): CTA j owns the tile-aligned shard j and
// computes its tiles' partials; each row's
// shards meet in the shared memory of one CTA, the row's folder, which folds
// all num_tiles partials in index order and returns the LSE to the others
// (the on-chip analogue of the pages' gather), so the result does not depend
// on virtual_tp.
//
// Layout of work.  Cluster q handles rows q, q + G, q + 2G, ... (G clusters).
// Within a CTA, 12 or 16 consumer warps reduce tiles (one warp per tile), one warp
// runs the exchange and fold, and one or two producer warps stream each item
// (one row's chunk of consecutive tiles, its 16-byte-aligned column span)
// into a ring slot with a 1-D bulk copy (cp.async.bulk, completion on the
// slot's "full" mbarrier).  Within a
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

#include <cstddef>
#include <cstdio>
#include <cstdlib>
#include <initializer_list>
#include <mutex>
#include <string>

#include "rlk_fold.cuh"
#include "rlk_internal.h"
#include "rlk_ptx.cuh"

namespace rlk {
namespace {

// Warps of a CTA: NW consumer warps (0 .. NW-1), the fold warp (NW), then the
// producer warps.  Measured on GB300 (same-box sweeps of 4-30 consumer warps):
//  * one CTA per SM: 16 consumer warps, two producers (one thread's bulk-copy
//    issue rate does not keep up with HBM);
//  * two CTAs per SM, one producer each: 12 consumer warps -- they fit the
//    halved register budget (72 registers) without spilling; 16 spilled and
//    ran up to 40% slower, and for the fused L2 schedule 8 warps ran 1.5%
//    slower at virtual TP 8 and 4 warps 32% slower.
__host__ __device__ constexpr int consumers_for(int mode, int per_sm) {
    return per_sm == 1 ? 16 : 12;
}
__host__ __device__ constexpr int producers_for(int per_sm) { return per_sm == 1 ? 2 : 1; }
__host__ __device__ constexpr int threads_for(int mode, int per_sm) {
    return (consumers_for(mode, per_sm) + 1 + producers_for(per_sm)) * 32;
}

constexpr int kMaxSlots = 96;
constexpr uint64_t kDrainNs = 1000000000ull;   // bound of the final drain of own copies
constexpr int64_t kL2ReuseBytes = 64ll << 20;  // logits held in L2 between the two reads of kModeFusedL2
constexpr int kMaxSkew = 2;  // measured at virtual TP 8: skew 1-2 beat 3-4
constexpr int kMinSlotsShared = 4;  // fewest ring slots worth running two CTAs per SM
constexpr int64_t kFusedChunkCols = 16384;

// Variants of a kernel, as template flags so that a launch without them runs
// none of their code (each adds code the fused kernel measured slower with).
constexpr int kFlagEnt = 1;   // the entropy of each row's softmax
constexpr int kFlagGrpo = 2;  // the fused GRPO step: g formed on chip (kModeFusedL2)
// Unrolling of the tile loops in the GRPO instantiations (4 elsewhere).  Their
// larger code stalls on instruction fetch at two CTAs per SM; measured at
// virtual TP 8 (65536 x 152576): unroll 2 6.45 ms against 6.76 with 4, while
// unroll 2 made the plain kernels slower (forward TP 1 2.80 against 2.72 ms,
// TP 8 3.38 against 3.17, fused TP 8 6.42 against 6.39).
constexpr int kTileUnrollGrpo = 2;
// Unrolling of the fold's 64-step recurrence in the fused L2 schedule without
// the entropy (64 elsewhere).  The same bits; measured at 65536 x 152576 (same
// box): fused TP 8 6.33 ms against 6.39 fully unrolled, TP 4 6.16 against
// 6.14, TP 1-2 unchanged; the forward at TP 8 (3.30 against 3.17 ms) and the
// entropy paths got slower with 8, and choosing by cluster size at run time
// (both folds in the kernel) made the GRPO step at TP 8 slower (6.51 ms).
constexpr int kFoldUnrollFusedL2 = 8;

struct SlotHdr {  // row metadata the producer writes beside each slot
    int64_t target;
    float g;
    float lse_in;
    int32_t active;
    int32_t pad;
    int64_t row;
};
static_assert(sizeof(SlotHdr) == 32, "SlotHdr layout");

struct RowShared {  // per-row state of the fold, one per row buffer
    int64_t target;
    float g;         // the header's g (the advantage A_r in the GRPO step)
    int16_t active;  // (written by the warp of the row's first tile ...
    int16_t has_xt;  //  ... and by the warp of the target's tile: separate halves of one word)
    float xt;        // f32(logit[row, target]) when this CTA owns the target's tile
    float ref;       // GRPO step: the row's reference logp (the header's lse_in)
    float lse;       // from the fold: the row's LSE ...
    float gf;        // ... and, in the GRPO step, its g (one 8-byte remote store with lse)
};
static_assert(sizeof(RowShared) == 32, "RowShared layout");
static_assert(offsetof(RowShared, gf) == offsetof(RowShared, lse) + 4 && offsetof(RowShared, lse) % 8 == 0,
              "lse and gf travel as one 8-byte store");

// Division by a divisor fixed for the launch (Granlund and Montgomery,
// "Division by invariant integers using multiplication", 1994): with
// s = ceil(log2 d) and m = floor(2^32 (2^s - d) / d) + 1, n / d equals
// (umulhi(n, m) + n) >> s for every 32-bit n (the sum taken in 33 bits).
struct FastDiv {
    uint32_t d, m, s;
};

__device__ __forceinline__ uint32_t fdiv(uint32_t n, const FastDiv& f) {
    return (uint32_t)(((uint64_t)__umulhi(n, f.m) + n) >> f.s);
}

struct Params {
    StreamArgs a;
    int64_t T, Vr, Vp, stride, ignore_index;
    uint64_t wait_ns;
    int32_t NT, W, C, mask_mode, NS, slot_bytes;
    int32_t tps;  // tiles per ring slot (consecutive tiles of one row share a slot when narrow)
    FastDiv ns_div;  // division by NS
    int32_t rbufs, rb_shift;  // row buffers of the fold (a power of two) and its log2
    int32_t skew;             // kModeFusedL2: phase A runs `skew` rows ahead of phase B (< rbufs)
    int32_t ent;  // the launch computes the entropy (stream_kernel's kFlagEnt)
    int32_t row_skip;  // kModeFwd, kModeFusedL2: consumer warps skip the rows in which they have no tile (row_skip_safe)
    uint32_t off_full, off_empty, off_hdr, off_seq, off_part, off_fold, off_rows, off_xtin, off_bars, off_flag;
    uint32_t off_meta;  // TileMeta of each of the CTA's tiles
    uint32_t off_tpart, off_foldt;  // ENT: t_k per row buffer, and the fold's scratch for them
};

// Columns fit in 32 bits: V_padded = num_tiles * W <= 1024 * 16384.
struct TileGeom {
    int ts, te;  // tile columns [ts, te)
    int hi;      // min(te, V_real): end of the tile's real columns
    int a;       // floor8(ts): column of the tile's first 8-column group
    int b;       // end of the data held in shared memory (multiple of 8)
};

// Columns [a, b) of tiles [kf, kl) that one ring slot holds:
// a = floor8(kf*W), b = min(ceil8(kl*W), floor8(V_real)); b <= a means nothing to copy.
struct Span {
    int a, b;
};

__device__ __forceinline__ Span chunk_span(int kf, int kl, const Params& p) {
    Span s;
    s.a = (kf * p.W) & ~7;
    const int ce = (kl * p.W + 7) & ~7;
    const int fv = (int)p.Vr & ~7;
    s.b = ce < fv ? ce : fv;
    return s;
}

// Geometry of tile k inside a slot that holds columns [sp.a, sp.b).
__device__ __forceinline__ TileGeom tile_geom(int k, const Params& p, const Span& sp) {
    TileGeom t;
    t.ts = k * p.W;
    t.te = t.ts + p.W;
    t.hi = t.te < (int)p.Vr ? t.te : (int)p.Vr;
    t.a = t.ts & ~7;
    t.b = sp.b;
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
    // Bounded wait until a shared-memory word equals `want`.
    __device__ bool wait_value(const volatile uint32_t* addr, uint32_t want) const {
        if (*addr == want) return true;
        if (*abort_flag) return false;
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
            if (*addr == want) return true;
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

// A plain, coherent global load.  The backward may write dlogits over the
// logits it reads (in place), so no read of the logits goes through the
// read-only data path, whose contents must not change during a kernel.
__device__ __forceinline__ uint16_t ld_bf16(const uint16_t* p) { return *p; }

// The 8 BF16 values of columns [c0, c0+8) as a uint4; columns outside the
// tile's real range [ts, hi) read as -inf.  Groups inside the slot span come
// from shared memory; the ragged real tail [floor8(V_real), V_real) is read
// from global memory one element at a time.
__device__ __forceinline__ uint4 load_group(const uint16_t* slot, const uint16_t* grow, int c0,
                                            const TileGeom& t) {
    uint4 v;
    if (c0 + 8 <= t.b) {
        v = *reinterpret_cast<const uint4*>(slot + (c0 - t.a));
    } else {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = c0 + 2 * j;
            const uint32_t lo = (c < t.hi && c >= t.ts) ? ld_bf16(grow + c) : 0xFF80u;
            const uint32_t hi = (c + 1 < t.hi && c + 1 >= t.ts) ? ld_bf16(grow + c + 1) : 0xFF80u;
            w[j] = lo | (hi << 16);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (c0 < t.ts || c0 + 8 > t.hi) {
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = c0 + 2 * j;
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

// Groups of one tile, indexed from floor8(ts): the "interior" groups [lo, hi)
// lie entirely inside [ts, min(end, floor8(V_real))) -- full, real, and always
// held in the slot -- and take a branch-free path; the others (a partial first
// group, a partial last group, the real tail) are "edges".  The split depends
// only on the tile and V_real, never on how tiles are grouped into slots.
struct GroupRange {
    int lo, hi, n;  // interior [lo, hi), all groups [0, n)
};

__device__ __forceinline__ GroupRange group_range(const TileGeom& t, int end, int Vr) {
    GroupRange g;
    g.lo = (t.ts > t.a) ? 1 : 0;
    const int fv = Vr & ~7;
    const int lim = end < fv ? end : fv;
    const int hi = (lim - t.a) >> 3;
    g.n = (((end + 7) & ~7) - t.a) >> 3;
    g.hi = hi < g.lo ? g.lo : hi;
    if (g.hi > g.n) g.hi = g.n;
    return g;
}

__device__ __forceinline__ int edge_group(const GroupRange& g, int e) { return e < g.lo ? 0 : g.hi + (e - g.lo); }

// Constants of tile l of a CTA's shard (global tile k0 + l), the same for
// every row: computed once per launch into shared memory.
struct __align__(16) TileMeta {
    TileGeom g;      // columns, in the slot that holds the tile's chunk
    int c;           // chunk of the tile: l / tps
    int share;       // arrivals the tile owes its slot's empty barrier
    int soff;        // elements from the slot's start to the tile's first group
    GroupRange ga;   // groups of the partial (real columns)
    int nb;          // groups of the gradient (all the tile's columns)
};
static_assert(sizeof(TileMeta) == 48, "TileMeta layout");

// A slot's empty barrier expects tps arrivals: the last tile of a short
// (end-of-row) chunk arrives for the missing tiles too.
__device__ void fill_meta(const Params& p, int k0, int ntl, TileMeta* meta) {
    for (int l = threadIdx.x; l < ntl; l += blockDim.x) {
        const int c = l / p.tps;
        const int kf = k0 + c * p.tps;
        const int kl = min(kf + p.tps, k0 + ntl);
        const Span sp = chunk_span(kf, kl, p);
        TileMeta m;
        m.g = tile_geom(k0 + l, p, sp);
        m.c = c;
        m.share = (k0 + l == kl - 1) ? 1 + p.tps - (kl - kf) : 1;
        m.soff = m.g.a - sp.a;
        m.ga = group_range(m.g, m.g.hi, (int)p.Vr);
        m.nb = group_range(m.g, m.g.te, (int)p.Vr).n;
        meta[l] = m;
    }
}

__device__ __forceinline__ void max4(uint32_t (&acc)[4], const uint4& v) {
    acc[0] = bf16x2_max_nan(acc[0], v.x);
    acc[1] = bf16x2_max_nan(acc[1], v.y);
    acc[2] = bf16x2_max_nan(acc[2], v.z);
    acc[3] = bf16x2_max_nan(acc[3], v.w);
}

// The two BF16 values of a packed word as an FP32 pair (lo, hi).
__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t w) {
    return make_float2(bf16lo_to_f32(w), bf16hi_to_f32(w));
}

// 2^(x*log2e + c) of an FP32 pair: one packed FMA (each lane rounded as a
// scalar FMA would be) and two SFU exponentials.
__device__ __forceinline__ float2 exp_terms2(float2 x, float2 c) {
    const float2 t = ffma2(x, make_float2(kLog2e, kLog2e), c);
    return make_float2(ex2_approx(t.x), ex2_approx(t.y));
}

// Accumulates the 8 exp terms of a group into 4 packed accumulators:
// s[j] holds the running sums of elements 2j and 2j+1 of every group.
__device__ __forceinline__ void sum8(float2 (&s)[4], const uint4& v, float nmL) {
    const float2 c = make_float2(nmL, nmL);
    s[0] = fadd2(s[0], exp_terms2(bf16x2_to_f32x2(v.x), c));
    s[1] = fadd2(s[1], exp_terms2(bf16x2_to_f32x2(v.y), c));
    s[2] = fadd2(s[2], exp_terms2(bf16x2_to_f32x2(v.z), c));
    s[3] = fadd2(s[3], exp_terms2(bf16x2_to_f32x2(v.w), c));
}

// sum8 plus t[j] += e x for the same terms (the tile's sum_c e^(x_c - m) x_c).
// A -inf column (padding, masked edges, or a -inf logit) must add 0 to t, not
// 0 * -inf.  CLAMP: the pair is first clamped to the largest finite negative
// BF16 (max.NaN keeps a NaN); its term e stays exactly 0 (x log2e overflows
// to -inf), so s is bitwise that of sum8.  Without CLAMP a finite pair gives
// the same bits, and a -inf one makes t NaN (tile_partial then redoes the
// tile with CLAMP).
template <bool CLAMP>
__device__ __forceinline__ void sum8_ent(float2 (&s)[4], float2 (&t)[4], const uint4& v, float nmL) {
    const float2 c = make_float2(nmL, nmL);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 x = bf16x2_to_f32x2(CLAMP ? bf16x2_max_nan(w[j], 0xFF7FFF7Fu) : w[j]);
        const float2 e = exp_terms2(x, c);
        s[j] = fadd2(s[j], e);
        t[j] = ffma2(e, x, t[j]);
    }
}

__device__ __forceinline__ float combine8(const float2 (&a)[4]) {
    return __fadd_rn(__fadd_rn(__fadd_rn(a[0].x, a[0].y), __fadd_rn(a[1].x, a[1].y)),
                     __fadd_rn(__fadd_rn(a[2].x, a[2].y), __fadd_rn(a[3].x, a[3].y)));
}

// (m_k, s_k) of one tile, computed by one warp; every lane returns the same value.
// Lane l visits interior groups lo+l, lo+l+32, ... then its edge groups; the
// tile maximum is exact, the sum uses 8 accumulators combined pairwise, then
// a fixed xor butterfly across lanes.  ENT: also t_k = sum_c e^(x_c - m_k) x_c
// into *t_out, accumulated beside s in the same order (s is unchanged).
//
// ENT_CLAMP (ENT only): clamp every pair, interior groups too.  Otherwise
// interior groups skip the clamp and the rare tile whose t comes out NaN is
// redone clamped; both give the same bits.  Measured on GB300: skipping it
// speeds the forward with entropy by 2-3.5% and slows the fused schedule's
// larger kernel by 4-6%, so the fused schedule clamps everywhere.
//
// UNROLL: of the interior loops.  Each lane adds its groups in the same order
// whatever the unrolling, so the bits do not depend on it; it trades loop
// overhead against code size (see kTileUnrollGrpo).
template <bool ENT, bool ENT_CLAMP = true, int UNROLL = 4>
__device__ float2 tile_partial(const uint16_t* slot, const uint16_t* grow, const TileGeom& t, const GroupRange& gr,
                               int lane, float* t_out) {
    if (ENT) *t_out = 0.f;
    if (t.hi <= t.ts) return make_float2(-INFINITY, 0.f);  // padding-only tile: identity
    const int ne = gr.lo + (gr.n - gr.hi);
    const uint4* s4 = reinterpret_cast<const uint4*>(slot);
    uint32_t acc[4] = {0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u};
#pragma unroll UNROLL
    for (int gi = gr.lo + lane; gi < gr.hi; gi += 32) max4(acc, s4[gi]);
    for (int e = lane; e < ne; e += 32) max4(acc, load_group(slot, grow, t.a + 8 * edge_group(gr, e), t));
    acc[0] = bf16x2_max_nan(bf16x2_max_nan(acc[0], acc[1]), bf16x2_max_nan(acc[2], acc[3]));
    const float m = warp_max_nan(fmax_nan(bf16lo_to_f32(acc[0]), bf16hi_to_f32(acc[0])));
    if (m == -INFINITY) return make_float2(-INFINITY, 0.f);  // all -inf: identity
    const float nmL = -__fmul_rn(m, kLog2e);
    float2 sm[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
    if constexpr (!ENT) {
#pragma unroll UNROLL
        for (int gi = gr.lo + lane; gi < gr.hi; gi += 32) sum8(sm, s4[gi], nmL);
        for (int e = lane; e < ne; e += 32)
            sum8(sm, load_group(slot, grow, t.a + 8 * edge_group(gr, e), t), nmL);
        return make_float2(m, warp_sum(combine8(sm)));
    } else {
        // Without ENT_CLAMP interior groups (real logits only) skip the
        // clamp, which only a -inf logit needs.  Edge groups (masked columns
        // read as -inf) always clamp.
        float2 tm[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll UNROLL
        for (int gi = gr.lo + lane; gi < gr.hi; gi += 32) sum8_ent<ENT_CLAMP>(sm, tm, s4[gi], nmL);
        for (int e = lane; e < ne; e += 32)
            sum8_ent<true>(sm, tm, load_group(slot, grow, t.a + 8 * edge_group(gr, e), t), nmL);
        float tk = warp_sum(combine8(tm));
        if (!ENT_CLAMP && __builtin_expect(isnan(tk), 0) && !isnan(m)) {
            // t is NaN but no logit is: a -inf logit met 0 * -inf.  Redo the
            // tile with every pair clamped (the same operations in the same
            // order as the fast path wherever a pair is finite).
#pragma unroll
            for (int j = 0; j < 4; ++j) sm[j] = tm[j] = make_float2(0.f, 0.f);
            for (int gi = gr.lo + lane; gi < gr.hi; gi += 32) sum8_ent<true>(sm, tm, s4[gi], nmL);
            for (int e = lane; e < ne; e += 32)
                sum8_ent<true>(sm, tm, load_group(slot, grow, t.a + 8 * edge_group(gr, e), t), nmL);
            tk = warp_sum(combine8(tm));
        }
        *t_out = tk;
        return make_float2(m, warp_sum(combine8(sm)));
    }
}

// dlogits of 8 columns from their exp terms: -g * p, and g * (1 - p) at
// column e of the group (the target), if 0 <= e < 8.
__device__ __forceinline__ uint4 grad8(const float (&pr)[8], int e, float g) {
    float d[8];
    const float2 ng2 = make_float2(-g, -g);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const float2 q = fmul2(make_float2(pr[e], pr[e + 1]), ng2);
        d[e] = q.x;
        d[e + 1] = q.y;
    }
    if ((unsigned)e < 8u) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j == e) d[j] = __fmul_rn(g, __fsub_rn(1.f, pr[j]));
    }
    return make_uint4(pack_bf16x2_rn(d[0], d[1]), pack_bf16x2_rn(d[2], d[3]), pack_bf16x2_rn(d[4], d[5]),
                      pack_bf16x2_rn(d[6], d[7]));
}

// dlogits of one tile's columns [ts, te) of one row, by one warp.
__device__ void tile_grad(const uint16_t* slot, const uint16_t* grow, uint16_t* drow, const TileGeom& t,
                          const GroupRange& gr, int Vr, bool active, int64_t target, float g, float lse, int lane) {
    const int ne = gr.lo + (gr.n - gr.hi);
    uint4* d4 = reinterpret_cast<uint4*>(drow + t.a);
    if (!active) {
        for (int gi = gr.lo + lane; gi < gr.hi; gi += 32) __stcs(d4 + gi, make_uint4(0u, 0u, 0u, 0u));
        for (int e = lane; e < ne; e += 32) {
            const int c0 = t.a + 8 * edge_group(gr, e);
            for (int j = 0; j < 8; ++j) {
                const int c = c0 + j;
                if (c >= t.ts && c < t.te) drow[c] = 0;
            }
        }
        return;
    }
    const float nlL = -__fmul_rn(lse, kLog2e);
    // the target's column relative to the tile's first group (-1: not in this tile)
    const int trel = (target >= t.ts && target < t.hi) ? (int)(target - t.a) : -1;
    const int tg_gi = trel >> 3, tg_e = trel & 7;
    const uint4* s4 = reinterpret_cast<const uint4*>(slot);
#pragma unroll 2
    for (int gi = gr.lo + lane; gi < gr.hi; gi += 32) {
        const uint4 v = s4[gi];
        const float2 c = make_float2(nlL, nlL);
        const float2 p0 = exp_terms2(bf16x2_to_f32x2(v.x), c), p1 = exp_terms2(bf16x2_to_f32x2(v.y), c);
        const float2 p2 = exp_terms2(bf16x2_to_f32x2(v.z), c), p3 = exp_terms2(bf16x2_to_f32x2(v.w), c);
        const float pr[8] = {p0.x, p0.y, p1.x, p1.y, p2.x, p2.y, p3.x, p3.y};
        __stcs(d4 + gi, grad8(pr, gi == tg_gi ? tg_e : -1, g));
    }
    for (int e = lane; e < ne; e += 32) {
        const int c0 = t.a + 8 * edge_group(gr, e);
        float pr[8];
        if (c0 + 8 <= t.b) {
            const uint4 v = *reinterpret_cast<const uint4*>(slot + (c0 - t.a));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 q = exp_terms2(bf16x2_to_f32x2(w[j]), make_float2(nlL, nlL));
                pr[2 * j] = q.x;
                pr[2 * j + 1] = q.y;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                const int c = c0 + j;
                const uint32_t lo = (c < Vr) ? ld_bf16(grow + c) : 0xFF80u;
                const uint32_t hi = (c + 1 < Vr) ? ld_bf16(grow + c + 1) : 0xFF80u;
                const float2 q = exp_terms2(bf16x2_to_f32x2(lo | (hi << 16)), make_float2(nlL, nlL));
                pr[j] = q.x;
                pr[j + 1] = q.y;
            }
        }
        uint4 q = grad8(pr, trel - (c0 - t.a), g);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = c0 + j;
            if (c >= t.ts && c < t.te)
                drow[c] = (c >= Vr) ? (uint16_t)0 : (uint16_t)((j & 1) ? (w[j >> 1] >> 16) : (w[j >> 1] & 0xFFFFu));
        }
    }
}

// ----------------------------------------------------------------- kernel roles

// Per-row buffers of the fold: row n uses buffer n % rbufs, and its
// mbarriers complete once per use, so a wait for row n takes parity
// (n / rbufs) & 1.
constexpr int kMaxRowBufs = 8;
constexpr int kMaxCluster = 8;

__device__ __forceinline__ int row_buf(const Params& p, int64_t n) { return (int)(n & (p.rbufs - 1)); }
__device__ __forceinline__ uint32_t row_par(const Params& p, int64_t n) { return (uint32_t)((n >> p.rb_shift) & 1); }

struct Ctx {
    int warp, lane;
    uint32_t rank;
    int64_t q, G, nrows;
    int k0, ntl, nch;  // first tile, tiles and ring chunks of this CTA per row
    unsigned char* smem;
    uint32_t sbase, full0, empty0;
    // per row buffer b: rowdone[b] (every consumer warp arrived: partials of the
    // row are in part[b]), lseready[b] (rows[b].lse valid), partfree[b]
    // (part[b] and rows[b] may be reused), xbar[b] (the folder: every peer's
    // partials and target record arrived), lsebar[b] (the others: the
    // folder's LSE arrived)
    uint32_t rowdone0, lseready0, partfree0, xbar0, lsebar0;
    SlotHdr* hdr;
    // seq[s]: number of the item the producer last issued into slot s.  A
    // consumer waits for its own item number before the slot's full-barrier
    // parity, so it never waits more than one phase ahead (a parity wait two
    // phases ahead would report a completion that has not happened).
    volatile uint32_t* seq;
    float2* part;
    float2* fold;
    RowShared* rows;
    float2* xtin;  // [rbufs][kMaxCluster]: each peer's (x_t, has_xt) of the row this CTA folds
    float* tpart;  // ENT: [rbufs][NT] t_k = sum_c e^(x_c - m_k) x_c beside part
    float* foldt;  // ENT: [NT] fold scratch
    const TileMeta* meta;  // [ntl] per-tile constants
    Waiter wt;
};

// Position of an item in the slot ring: slot index and the parity of the pass.
struct RingPos {
    int slot;
    uint32_t par;
};


// The producer issues blocks of nch items (one row's chunks for one phase).
// kModeFwd / kModeBwd / kModeFused: block n is row n.  kModeFusedL2 with
// skew S follows the consumers' order: A(0), ..., A(S-1), then A(n+S), B(n)
// for n = 0, 1, ... (A(n+S) only while n+S < R).  With S0 = min(S, R) and
// P = max(R - S, 0) full pairs: A(n) is block n for n < S0 and S0 + 2(n-S)
// after; B(n) is block S0 + 2n + 1 for n < P and S0 + 2P + (n - P) after.
__device__ __forceinline__ int64_t block_of(int MODE, int64_t n, bool phase_b, int64_t R, int64_t S) {
    if (MODE != kModeFusedL2) return n;
    const int64_t S0 = S < R ? S : R;
    const int64_t P = R > S ? R - S : 0;
    if (!phase_b) return n < S0 ? n : S0 + 2 * (n - S);
    return n < P ? S0 + 2 * n + 1 : S0 + 2 * P + (n - P);
}

// Inverse of block_of for kModeFusedL2: block j -> (row, is phase B).
__device__ __forceinline__ void block_row(int64_t j, int64_t R, int64_t S, int64_t& n, bool& phase_b) {
    const int64_t S0 = S < R ? S : R;
    const int64_t P = R > S ? R - S : 0;
    if (j < S0) {
        n = j;
        phase_b = false;
        return;
    }
    const int64_t jj = j - S0;
    if (jj < 2 * P) {
        phase_b = (jj & 1) != 0;
        n = phase_b ? jj / 2 : jj / 2 + S;
    } else {
        phase_b = true;
        n = P + (jj - 2 * P);
    }
}

__device__ __forceinline__ RingPos ring_of(uint32_t item, const FastDiv& ns) {
    const uint32_t q = fdiv(item, ns);
    return RingPos{(int)(item - q * ns.d), q & 1u};
}

// Row metadata of 32 consecutive rows of this CTA, one row per lane.
struct MetaWindow {
    int64_t t = 0;
    int32_t act = 0;
    float g = 0.f, lin = 0.f;
};

// Producer warp pid of NP issues the items i with i mod NP == pid, in order.
// Before the parity wait on a slot's empty barrier it waits until the slot
// holds item i - NS: with several producers the slot's previous item may
// belong to another one, and a parity wait while that item is not yet
// issued could pass two phases ahead and overwrite a slot still in use.
template <int MODE, int NP, int F>
__device__ void producer(const Params& p, const Ctx& x, int pid) {
    constexpr bool GRPO = (F & kFlagGrpo) != 0;
    const int lane = x.lane;
    const uint64_t pol_first = l2_policy_evict_first();
    const uint64_t pol_last = l2_policy_evict_last();
    // Windows [base, base+32) and [base-32, base): kModeFusedL2 visits row n
    // after row n+1, which can lie in the next window.
    int64_t meta_base = 0;
    MetaWindow cur, prev;
    auto load_meta = [&](int64_t base) {
        const int64_t n = base + lane;
        if (n < x.nrows) {
            const int64_t r = x.q + n * x.G;
            cur.t = p.a.targets[r];
            cur.act = (p.mask_mode == RLK_MASK_EXPLICIT) ? (p.a.mask[r] != 0) : (cur.t != p.ignore_index);
            if (GRPO) {  // the GRPO step: A_r and ref_r ride in g and lse_in
                cur.g = p.a.adv[r];
                cur.lin = p.a.ref ? p.a.ref[r] : 0.f;
            } else {
                cur.g = (MODE != kModeFwd) ? p.a.grad[r] : 0.f;
                cur.lin = (MODE == kModeBwd) ? p.a.lse_in[r] : 0.f;
            }
        }
    };
    load_meta(0);
    int64_t issued = 0;
    int slot = 0;
    uint32_t phase = 0;
    bool aborted = false;
    const int64_t nblocks = (MODE == kModeFusedL2) ? 2 * x.nrows : x.nrows;
    for (int64_t j = 0; j < nblocks && !aborted; ++j) {
        int64_t n = j;
        bool second = false;  // kModeFusedL2: the phase-B copy of row n
        if (MODE == kModeFusedL2) block_row(j, x.nrows, p.skew, n, second);
        if (n - meta_base >= 32) {
            prev = cur;
            meta_base += 32;
            load_meta(meta_base);
        }
        const bool in_cur = n >= meta_base;
        const int src = (int)(in_cur ? n - meta_base : n - meta_base + 32);
        const int64_t t_c = (int64_t)__shfl_sync(0xFFFFFFFFu, (unsigned long long)cur.t, src);
        const int64_t t_p = (int64_t)__shfl_sync(0xFFFFFFFFu, (unsigned long long)prev.t, src);
        const int32_t a_c = __shfl_sync(0xFFFFFFFFu, cur.act, src), a_p = __shfl_sync(0xFFFFFFFFu, prev.act, src);
        const float g_c = __shfl_sync(0xFFFFFFFFu, cur.g, src), g_p = __shfl_sync(0xFFFFFFFFu, prev.g, src);
        const float l_c = __shfl_sync(0xFFFFFFFFu, cur.lin, src), l_p = __shfl_sync(0xFFFFFFFFu, prev.lin, src);
        const int64_t t = in_cur ? t_c : t_p;
        const int32_t act = in_cur ? a_c : a_p;
        const float g = in_cur ? g_c : g_p;
        const float lin = in_cur ? l_c : l_p;
        // Which copies move bytes, and their L2 hint: an inactive row's
        // columns are needed by phase A only; the first copy of a row that
        // kModeFusedL2 reads again stays in L2 (evict-last).
        const bool needs_bytes = !((MODE == kModeBwd || second) && !act);
        const uint64_t policy = (MODE == kModeFusedL2 && !second && act) ? pol_last : pol_first;
        const int64_t row = x.q + n * x.G;
        const uint16_t* grow = p.a.logits + row * p.stride;
        for (int c = 0; c < x.nch; ++c) {
            const bool mine = NP == 1 || (int)(issued % NP) == pid;
            bool ok = true;
            if (lane == 0 && mine) {
                if (NP > 1 && issued >= p.NS) ok = x.wt.wait_value(x.seq + slot, (uint32_t)(issued - p.NS));
                if (ok) ok = x.wt.wait(x.empty0 + 8u * slot, phase ^ 1u, false);
            }
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) {
                aborted = true;
                break;
            }
            if (lane == 0 && mine) {
                SlotHdr h;
                h.target = t;
                h.g = g;
                h.lse_in = lin;
                h.active = act;
                h.pad = 0;
                h.row = row;
                x.hdr[slot] = h;
                x.seq[slot] = (uint32_t)issued;
                const int kf = x.k0 + c * p.tps;
                const int kl = min(kf + p.tps, x.k0 + x.ntl);
                const Span sp = chunk_span(kf, kl, p);
                const uint32_t bytes = (sp.b > sp.a && needs_bytes) ? (uint32_t)((sp.b - sp.a) * 2) : 0u;
                const uint32_t fb = x.full0 + 8u * slot;
                if (bytes) {
                    mbar_arrive_expect_tx(fb, bytes);
                    bulk_g2s(x.sbase + (uint32_t)slot * (uint32_t)p.slot_bytes, grow + sp.a, bytes, fb, policy);
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
    // Drain: wait (bounded) until every copy this warp issued has landed.
    if (lane == 0) {
        const int64_t first = issued > p.NS ? issued - p.NS : 0;
        for (int64_t j = first; j < issued; ++j) {
            if (NP > 1 && (int)(j % NP) != pid) continue;
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

// The fold warp.  Row n of a cluster is folded by one CTA, its folder
// F(n) = n mod C (every row by the CTA itself when C = 1).
//  * push (row order, once every consumer warp has put its tiles' partials in
//    part[b]): a CTA that does not fold the row sends its shard of partials
//    and its target record (x_t, has_xt) to the folder with asynchronous
//    remote stores, which complete on the folder's xbar[b]; the folder arms
//    xbar[b] with the bytes it expects (one local arrival with expect-tx).
//    Every CTA arrives once per row on xbar[b] and lsebar[b] (with expect-tx
//    where it receives), so both have one phase per row.
//  * fold (this CTA's rows, in order, as soon as xbar[b] completes): fold all
//    tiles in index order (fold_tiles), write LSE and logp, and send the LSE
//    to every other CTA (remote stores completing on their lsebar[b]).
//  * release (row order, once the row's LSE is here): rows[b].lse is valid
//    (lseready) and the row's buffers may be reused (partfree).
// The warp runs the three as an event loop with non-blocking tests, so a
// row's fold never waits for the LSE of an earlier row folded elsewhere; the
// only chain between rows is the reuse of a buffer: the push of row
// n + rbufs needs phase A of that row, which needs the release of row n,
// which needs row n's LSE, which its folder sends after its fold.  So no
// push of a later row can land in a buffer whose row is still being
// exchanged or folded.  Each test of a phase expects the barrier to have
// completed the phase of the previous use of its buffer, which the loop's
// order guarantees: rows are pushed, folded and released in increasing order.
__device__ __forceinline__ bool folds_row(const Params& p, const Ctx& x, int64_t n) {
    return p.C == 1 || (uint32_t)(n & (p.C - 1)) == x.rank;  // C is a power of two
}

__device__ __forceinline__ bool warp_test(uint32_t bar, uint32_t parity, bool cluster_scope) {
    const bool ok = cluster_scope ? mbar_test_wait_cluster(bar, parity) : mbar_test_wait(bar, parity);
    return __all_sync(0xFFFFFFFFu, ok);
}

template <int F>
__device__ void push_row(const Params& p, const Ctx& x, int64_t n) {
    constexpr bool ENT = (F & kFlagEnt) != 0, GRPO = (F & kFlagGrpo) != 0;
    if (p.C == 1) return;
    const int lane = x.lane;
    const int b = row_buf(p, n);
    const uint32_t xb = x.xbar0 + 8u * b, lb = x.lsebar0 + 8u * b;
    if (folds_row(p, x, n)) {
        // every peer's shard (all tiles but this CTA's own) and target record
        if (lane == 0) {
            mbar_arrive_expect_tx(xb, (uint32_t)((p.NT - x.ntl) * (ENT ? 12 : 8) + (p.C - 1) * 8));
            mbar_arrive(lb);
        }
        return;
    }
    const uint32_t f = (uint32_t)(n & (p.C - 1));
    const float2* part = x.part + (size_t)b * p.NT;
    const uint32_t fxb = mapa_shared(xb, f);
    for (int i = lane; i < x.ntl; i += 32) {
        const float2 v = part[x.k0 + i];
        st_async_f32x2(mapa_shared(smem_u32(&part[x.k0 + i]), f), v.x, v.y, fxb);
        if (ENT) {
            float* tp = x.tpart + (size_t)b * p.NT + x.k0 + i;
            st_async_f32(mapa_shared(smem_u32(tp), f), *tp, fxb);
        }
    }
    if (lane == 0) {
        RowShared& rs = x.rows[b];
        st_async_f32x2(mapa_shared(smem_u32(&x.xtin[b * kMaxCluster + x.rank]), f), rs.xt,
                       __int_as_float(rs.has_xt), fxb);
        rs.has_xt = 0;
        mbar_arrive(xb);
        mbar_arrive_expect_tx(lb, GRPO ? 8u : 4u);  // the folder's LSE (and, GRPO, the row's g)
    }
}

// g of a row in the fused GRPO step, in the GRPO loss kernel's FP32
// operations and order (so the two give the same bits): the row's advantage
// a, reference logp rf, logp lp and 1/N as FP32.  Not inlined: the fold warp
// calls it once per row, and a smaller kernel measured faster (0.2-0.4%).
__device__ __noinline__ float grpo_row_grad(const Params& p, bool active, float a, float rf, float lp,
                                               float inv_nf) {
    float dterm = -a;
    if (p.a.ref) {
        const float d = rf - lp;
        const float e = expf(d);
        dterm = fmaf(p.a.beta, 1.f - e, dterm);
    }
    return (active ? dterm : 0.f) * inv_nf;
}

template <int MODE, int F>
__device__ void fold_row(const Params& p, const Ctx& x, int64_t n, float inv_nf) {
    constexpr bool ENT = (F & kFlagEnt) != 0, GRPO = (F & kFlagGrpo) != 0;
    const int lane = x.lane;
    const int b = row_buf(p, n);
    float2* part = x.part + (size_t)b * p.NT;
    RowShared& rs = x.rows[b];
    float lse_v, ent_v = 0.f;
    if constexpr (ENT) {
        const float2 r = fold_tiles_ent(part, x.tpart + (size_t)b * p.NT, p.NT, x.fold, x.foldt, lane);
        lse_v = r.x;
        ent_v = r.y;
    } else {
        lse_v = fold_tiles<MODE == kModeFusedL2 ? kFoldUnrollFusedL2 : 64>(part, p.NT, x.fold, lane);
    }
    const int64_t row = x.q + n * x.G;
    if (p.a.partials) {
        float2* out = reinterpret_cast<float2*>(p.a.partials) + row * p.NT;
        for (int k = lane; k < p.NT; k += 32) out[k] = part[k];
    }
    // the target logit: captured here or sent by the CTA that owns its tile
    bool has = rs.has_xt != 0;
    float xt = rs.xt;
    if (p.C > 1) {
        const float2 r =
            lane < p.C && (uint32_t)lane != x.rank ? x.xtin[b * kMaxCluster + lane] : make_float2(0.f, 0.f);
        const unsigned from = __ballot_sync(0xFFFFFFFFu, __float_as_int(r.y) != 0);
        if (!has && from) {
            has = true;
            xt = __shfl_sync(0xFFFFFFFFu, r.x, __ffs(from) - 1);
        }
        // the LSE to every other CTA of the cluster
        if (!GRPO && lane < p.C && (uint32_t)lane != x.rank)
            st_async_f32(mapa_shared(smem_u32(&rs.lse), (uint32_t)lane), lse_v,
                         mapa_shared(x.lsebar0 + 8u * b, (uint32_t)lane));
    }
    const bool active = rs.active != 0;
    const int64_t t = rs.target;
    const bool in_range = t >= 0 && t < p.Vr;
    float gv = 0.f;
    if constexpr (GRPO) {
        // the row's logp and g (every lane), then the LSE and g to every other CTA
        const float lp = !active ? 0.f : (in_range && has) ? __fsub_rn(xt, lse_v) : __int_as_float(0x7FC00000);
        gv = grpo_row_grad(p, active, rs.g, rs.ref, lp, inv_nf);
        if (p.C > 1 && lane < p.C && (uint32_t)lane != x.rank)
            st_async_f32x2(mapa_shared(smem_u32(&rs.lse), (uint32_t)lane), lse_v, gv,
                           mapa_shared(x.lsebar0 + 8u * b, (uint32_t)lane));
    }
    __syncwarp();
    if (lane == 0) {
        p.a.lse[row] = lse_v;
        if (ENT) p.a.entropy[row] = ent_v;
        if (!active) {
            p.a.logp[row] = 0.f;
        } else if (!in_range) {
            p.a.logp[row] = __int_as_float(0x7FC00000);
            atomicOr(p.a.status, kStatusTargetRange);
        } else if (has) {
            p.a.logp[row] = __fsub_rn(xt, lse_v);
        }
        if (active && !isfinite(lse_v)) atomicOr(p.a.status, kStatusNonFinite);
        if (GRPO) {
            p.a.grad_out[row] = gv;
            rs.gf = gv;
        }
        rs.has_xt = 0;
        rs.lse = lse_v;
    }
    __syncwarp();
}

template <int MODE, int F>
__device__ void fold_warp(const Params& p, const Ctx& x) {
    // GRPO step: 1/N as FP32, formed as the GRPO loss kernel forms it
    float inv_nf = 0.f;
    if constexpr ((F & kFlagGrpo) != 0) {
        const unsigned long long n_act = *p.a.n_active;
        inv_nf = (float)(n_act > 0 ? 1.0 / (double)n_act : 0.0);
    }
    const int64_t R = x.nrows;
    int64_t np = 0, nr = 0;                         // next row to push, to release
    int64_t nf = p.C > 1 ? (int64_t)x.rank : 0;     // next row this CTA folds
    const int64_t fstep = p.C > 1 ? p.C : 1;
    bool idle = false;
    uint64_t t0 = 0;
    while (nr < R) {
        bool progressed = false;
        if (np < R && warp_test(x.rowdone0 + 8u * row_buf(p, np), row_par(p, np), false)) {
            push_row<F>(p, x, np);
            ++np;
            progressed = true;
        }
        if (nf < R && nf < np &&
            (p.C == 1 || warp_test(x.xbar0 + 8u * row_buf(p, nf), row_par(p, nf), true))) {
            fold_row<MODE, F>(p, x, nf, inv_nf);
            nf += fstep;
            progressed = true;
        }
        if (nr < np) {
            const int b = row_buf(p, nr);
            const bool ready =
                folds_row(p, x, nr) ? nr < nf : warp_test(x.lsebar0 + 8u * b, row_par(p, nr), true);
            if (ready) {
                if (x.lane == 0) {
                    if (MODE == kModeFused || MODE == kModeFusedL2) mbar_arrive(x.lseready0 + 8u * b);
                    mbar_arrive(x.partfree0 + 8u * b);
                }
                ++nr;
                progressed = true;
            }
        }
        if (progressed) {
            idle = false;
            continue;
        }
        // Every decision below is the same in all lanes: the clock is lane 0's.
        if (__any_sync(0xFFFFFFFFu, *x.wt.abort_flag != 0)) break;
        const uint64_t now = __shfl_sync(0xFFFFFFFFu, (unsigned long long)globaltimer_ns(), 0);
        if (!idle) {
            idle = true;
            t0 = now;
        } else if (now - t0 > x.wt.limit_ns) {
            if (x.lane == 0) {
                *x.wt.abort_flag = 1;
                atomicOr(x.wt.status, kStatusTimeout);
            }
            break;
        }
    }
    __syncwarp();
    // After an expired wait some peer stores may still be on their way into
    // this CTA's shared memory: give them time to land before the kernel ends.
    if (p.C > 1 && *x.wt.abort_flag) {
        const uint64_t t1 = globaltimer_ns();
        while (globaltimer_ns() - t1 < 1000000ull) {
        }
    }
}

// Work is per tile, copies are per chunk of tps tiles: consumer warp w
// takes the tiles l of row n with (n*ntl + l) mod W == w, waits on the full
// barrier of the tile's chunk, and releases its share of the chunk's slot
// when done.  A slot's empty barrier expects tps arrivals; the last tile of
// a short (end-of-row) chunk arrives for the missing tiles too.
struct TileItem {
    uint32_t item;   // number of the chunk's item in the producer's order
    int slot;
    uint32_t par;
};

// The item of a tile whose chunk is number c of a block whose first item is item0.
__device__ __forceinline__ TileItem tile_item(const Params& p, uint32_t item0, int c) {
    TileItem it;
    it.item = item0 + (uint32_t)c;
    const RingPos ps = ring_of(it.item, p.ns_div);
    it.slot = ps.slot;
    it.par = ps.par;
    return it;
}

// Waits (bounded, all 32 lanes) until the tile's slot holds item `item` and
// its bulk copy has landed.
__device__ __forceinline__ bool wait_item(const Ctx& x, const TileItem& it, uint32_t item) {
    const bool issued = __all_sync(0xFFFFFFFFu, x.wt.wait_value(x.seq + it.slot, item));
    const bool landed = x.wt.warp_wait(x.full0 + 8u * it.slot, it.par);
    if (!(issued && landed)) *x.wt.abort_flag = 1;
    return issued && landed;
}

// Guard of every tile: the slot's header must name the row this CTA expects.
// A slip of the ring protocol then stops the kernel with a status bit instead
// of addressing another row's memory.
__device__ __noinline__ void header_fail(uint32_t* status, volatile int* abort_flag) {
    atomicOr(status, kStatusInternal);
    *abort_flag = 1;
}

__device__ __forceinline__ bool header_ok(const Params& p, const Ctx& x, const SlotHdr& h, uint32_t want) {
    if (__builtin_expect((uint32_t)h.row == want, 1)) return true;  // rows of one launch differ in their low 32 bits
    if (x.lane == 0) header_fail(p.a.status, x.wt.abort_flag);
    return false;
}

// Consumer warp w of NW takes the tiles l of row n with (n*ntl + l) mod NW
// == w.  Rows come in order, so the rotation r = (n*ntl) mod NW advances by
// ntl mod NW per row.
template <int NW>
struct TileRotation {
    int r = 0, step = 0;
    __device__ explicit TileRotation(int ntl) : step(ntl % NW) {}
    // The first tile of this warp in the current row; moves to the next row.
    __device__ int next(int warp) {
        const int f = warp - r;
        r += step;
        if (r >= NW) r -= NW;
        return f < 0 ? f + NW : f;
    }
};

// Phase A of row n for one consumer warp: the partials of its tiles, the
// row metadata (tile 0) and the target logit (the tile that holds it).
// FWD releases each tile's share of its slot at once; FUSED keeps the slots
// for phase B.
template <int MODE, int W, int F>
__device__ bool phase_a(const Params& p, const Ctx& x, int64_t n, uint32_t item0, int first) {
    constexpr bool ENT = (F & kFlagEnt) != 0, GRPO = (F & kFlagGrpo) != 0;
    // With row_skip (the forward and the L2 fused schedule) a warp with no
    // tile in the row (ntl < NW) skips it: it writes nothing, and rowdone
    // counts only the min(NW, ntl) warps that have tiles.  Each of those
    // waits for partfree of row n - rbufs first; the planner allows the skip
    // only where that parity wait stays within one phase and, fused, where
    // the row's LSE outlives every phase B that reads it (row_skip_safe).
    // The resident fused schedule keeps every warp in every row.
    if ((MODE == kModeFwd || MODE == kModeFusedL2) && p.row_skip && first >= x.ntl) return true;
    const int lane = x.lane;
    const int b = row_buf(p, n);
    bool ok = true;
    if (n >= p.rbufs) ok = x.wt.warp_wait(x.partfree0 + 8u * b, row_par(p, n - p.rbufs));
    uint16_t* slots = reinterpret_cast<uint16_t*>(x.smem);
    const int slot_elems = p.slot_bytes / 2;
    const uint32_t want = (uint32_t)(x.q + n * x.G);
    for (int l = first; l < x.ntl && ok; l += W) {
        const TileMeta m = x.meta[l];
        const TileItem it = tile_item(p, item0, m.c);
        if (!wait_item(x, it, it.item)) {
            ok = false;
            break;
        }
        const SlotHdr h = x.hdr[it.slot];
        if (!header_ok(p, x, h, want)) {
            ok = false;
            break;
        }
        const uint16_t* grow = p.a.logits + h.row * p.stride;
        const int k = x.k0 + l;
        const TileGeom& tg = m.g;
        const uint16_t* sl = slots + (size_t)it.slot * slot_elems + m.soff;
        float tk = 0.f;
        const float2 pr =
            tile_partial<ENT, MODE != kModeFwd, GRPO ? kTileUnrollGrpo : 4>(sl, grow, tg, m.ga, lane, &tk);
        if (lane == 0) {
            RowShared& rs = x.rows[b];
            if (l == 0) {
                rs.target = h.target;
                rs.active = (int16_t)(h.active != 0);
                rs.g = h.g;
                if (GRPO) rs.ref = h.lse_in;
            }
            x.part[(size_t)b * p.NT + k] = pr;
            if (ENT) x.tpart[(size_t)b * p.NT + k] = tk;
            if (h.active && h.target >= tg.ts && h.target < tg.hi) {
                const uint16_t bits = (h.target < tg.b) ? sl[h.target - tg.a] : ld_bf16(grow + h.target);
                rs.xt = __uint_as_float((uint32_t)bits << 16);
                rs.has_xt = 1;
            }
        }
        if (MODE == kModeFwd || MODE == kModeFusedL2) {
            __syncwarp();
            if (lane == 0) mbar_arrive_n(x.empty0 + 8u * it.slot, (uint32_t)m.share);
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(x.rowdone0 + 8u * b);
    return ok;
}

// dlogits of row n's tiles for one consumer warp; each tile then releases its
// share of its slot.  FUSED: the slots are still resident from phase A and
// lse_v is the fold's LSE.  FUSED_L2: the tile waits for the second copy of
// its chunk; lse_v is the fold's LSE.  BWD: the tile waits for its chunk and
// reads the row's LSE (lse_in) from the slot header.
template <int MODE, int W, int F>
__device__ bool phase_b(const Params& p, const Ctx& x, int64_t n, uint32_t item0, float lse_v, float g_fold,
                        int first) {
    constexpr bool GRPO = (F & kFlagGrpo) != 0;
    constexpr bool kWaits = MODE == kModeBwd || MODE == kModeFusedL2;
    const int lane = x.lane;
    uint16_t* slots = reinterpret_cast<uint16_t*>(x.smem);
    const int slot_elems = p.slot_bytes / 2;
    const uint32_t want = (uint32_t)(x.q + n * x.G);
    for (int l = first; l < x.ntl; l += W) {
        const TileMeta m = x.meta[l];
        const TileItem it = tile_item(p, item0, m.c);
        if (kWaits && !wait_item(x, it, it.item)) return false;
        const SlotHdr h = x.hdr[it.slot];
        if (!header_ok(p, x, h, want)) return false;
        const TileGeom& tg = m.g;
        const float lse = (MODE == kModeBwd) ? h.lse_in : lse_v;
        if (MODE == kModeBwd && l == 0 && lane == 0 && h.active) {
            if (!p.a.foreign_targets && (h.target < 0 || h.target >= p.Vr)) atomicOr(p.a.status, kStatusTargetRange);
            if (!isfinite(h.lse_in)) atomicOr(p.a.status, kStatusNonFinite);
        }
        tile_grad(slots + (size_t)it.slot * slot_elems + m.soff, p.a.logits + h.row * p.stride,
                  p.a.dlogits + h.row * p.stride, tg, GroupRange{m.ga.lo, m.ga.hi, m.nb}, (int)p.Vr,
                  h.active != 0, h.target, GRPO ? g_fold : h.g, lse, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive_n(x.empty0 + 8u * it.slot, (uint32_t)m.share);
    }
    return true;
}

template <int MODE, int NW, int F>
__device__ void consumer(const Params& p, const Ctx& x) {
    const int64_t R = x.nrows;
    const uint32_t nch = (uint32_t)x.nch;
    const int64_t S = (MODE == kModeFusedL2) ? p.skew : 1;
    auto item_a = [&](int64_t n) { return (uint32_t)block_of(MODE, n, false, R, S) * nch; };
    auto item_b = [&](int64_t n) { return (uint32_t)block_of(MODE, n, MODE != kModeFused, R, S) * nch; };
    TileRotation<NW> rot_a(x.ntl), rot_b(x.ntl);  // phase A and phase B each visit rows in order
    if constexpr (MODE == kModeBwd) {
        for (int64_t n = 0; n < R; ++n)
            if (!phase_b<MODE, NW, F>(p, x, n, item_b(n), 0.f, 0.f, rot_b.next(x.warp))) break;
    } else if constexpr (MODE == kModeFwd) {
        for (int64_t n = 0; n < R; ++n) phase_a<MODE, NW, F>(p, x, n, item_a(n), rot_a.next(x.warp));
    } else {
        // Skewed order A(0), ..., A(S-1), then A(n+S), B(n): the fold of row
        // n overlaps phase A of rows n+1..n+S.  kModeFused (S = 1) keeps two
        // rows of slots resident; kModeFusedL2 copies each row a second time
        // for phase B.  rbufs > S keeps rows[b].lse of row n until every warp
        // has read it: row n + rbufs comes after B(n) in every warp's order.
        for (int64_t n = 0; n < S && n < R; ++n) phase_a<MODE, NW, F>(p, x, n, item_a(n), rot_a.next(x.warp));
        for (int64_t n = 0; n < R; ++n) {
            if (n + S < R) phase_a<MODE, NW, F>(p, x, n + S, item_a(n + S), rot_a.next(x.warp));
            const int b = row_buf(p, n);
            const int first_b = rot_b.next(x.warp);
            // row_skip: no tile in this row, so neither its LSE nor phase B
            if (MODE == kModeFusedL2 && p.row_skip && first_b >= x.ntl) continue;
            const bool ready = x.wt.warp_wait(x.lseready0 + 8u * b, row_par(p, n));
            // A failed wait anywhere sets the abort flag; the slot headers may
            // then be stale, so skip the writes (the status word already says
            // RLK_ERR_TIMEOUT).
            if (ready && !*x.wt.abort_flag)
                phase_b<MODE, NW, F>(p, x, n, item_b(n), x.rows[b].lse, (F & kFlagGrpo) ? x.rows[b].gf : 0.f,
                                     first_b);
        }
    }
}

// PER_SM: CTAs resident per SM (1 or 2); the register budget follows from it.
// F: kFlagEnt (the forward and the fused L2 schedule) also forms the entropy of
// each row's softmax; kFlagGrpo (the fused L2 schedule) is the GRPO step.
template <int MODE, int PER_SM, int F>
__global__ void __launch_bounds__(threads_for(MODE, PER_SM), PER_SM)
    stream_kernel(const __grid_constant__ Params p) {
    constexpr int NW = consumers_for(MODE, PER_SM);
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
    x.nch = (x.ntl + p.tps - 1) / p.tps;
    x.smem = smem;
    x.sbase = smem_u32(smem);
    x.full0 = x.sbase + p.off_full;
    x.empty0 = x.sbase + p.off_empty;
    x.rowdone0 = x.sbase + p.off_bars;
    x.lseready0 = x.rowdone0 + 8u * p.rbufs;
    x.partfree0 = x.lseready0 + 8u * p.rbufs;
    x.xbar0 = x.partfree0 + 8u * p.rbufs;
    x.lsebar0 = x.xbar0 + 8u * p.rbufs;
    x.hdr = reinterpret_cast<SlotHdr*>(smem + p.off_hdr);
    x.seq = reinterpret_cast<volatile uint32_t*>(smem + p.off_seq);
    x.part = reinterpret_cast<float2*>(smem + p.off_part);
    x.fold = reinterpret_cast<float2*>(smem + p.off_fold);
    x.rows = reinterpret_cast<RowShared*>(smem + p.off_rows);
    x.xtin = reinterpret_cast<float2*>(smem + p.off_xtin);
    x.tpart = reinterpret_cast<float*>(smem + p.off_tpart);
    x.foldt = reinterpret_cast<float*>(smem + p.off_foldt);
    x.meta = reinterpret_cast<const TileMeta*>(smem + p.off_meta);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + p.off_flag);
    x.wt.abort_flag = abort_flag;
    x.wt.status = p.a.status;
    x.wt.limit_ns = p.wait_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.NS; ++s) {
            mbar_init(x.full0 + 8u * s, 1);
            mbar_init(x.empty0 + 8u * s, (uint32_t)p.tps);
            x.seq[s] = 0xFFFFFFFFu;
        }
        for (int b = 0; b < p.rbufs; ++b) {
            mbar_init(x.rowdone0 + 8u * b,
                      (uint32_t)((MODE == kModeFwd || MODE == kModeFusedL2) && p.row_skip ? min(NW, x.ntl) : NW));
            mbar_init(x.lseready0 + 8u * b, 1);
            mbar_init(x.partfree0 + 8u * b, 1);
            mbar_init(x.xbar0 + 8u * b, 1);    // the local arrival (with expect-tx on the folder)
            mbar_init(x.lsebar0 + 8u * b, 1);  // the local arrival (with expect-tx off the folder)
            x.rows[b].has_xt = 0;
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    fill_meta(p, x.k0, x.ntl, reinterpret_cast<TileMeta*>(smem + p.off_meta));
    if (p.C > 1) cluster_sync_all(); else __syncthreads();

    if (x.warp > NW) {
        producer<MODE, producers_for(PER_SM), F>(p, x, x.warp - NW - 1);
    } else if (x.warp == NW) {
        if (MODE != kModeBwd) fold_warp<MODE, F>(p, x);
    } else {
        consumer<MODE, NW, F>(p, x);
    }

    __syncthreads();
    if (p.C > 1) cluster_sync_all();  // no CTA leaves while a peer may still write into it
}

// One warp waits, with the kernels' bounded wait, on an mbarrier that nothing
// arrives at; the wait must expire and record RLK_ERR_TIMEOUT.
__global__ void selftest_wait_kernel(uint32_t* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    Waiter wt{&abort_flag, status, limit_ns};
    wt.warp_wait(smem_u32(&bar), 0u);
    __syncthreads();
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

// Planner overrides, for measurement: RLK_CTAS_PER_SM (1 or 2), RLK_ROW_BUFS
// (2, 4 or 8), RLK_FUSED_SKEW (0 .. row buffers - 1) and RLK_FUSED_SCHEDULE
// (l2 or resident).  These are the ring shapes the host protocol model
// replays; any other value fails closed with RLK_ERR_UNSUPPORTED instead of
// being clamped, so no process can run a ring shape the model has not run.
rlk_status knob(const char* name, int dflt, std::initializer_list<int> allowed, int* out) {
    const char* v = std::getenv(name);
    *out = dflt;
    if (!v || !*v) return RLK_OK;
    char* end = nullptr;
    const long x = std::strtol(v, &end, 10);
    if (end && *end == '\0')
        for (int a : allowed)
            if (x == a) {
                *out = a;
                return RLK_OK;
            }
    return fail(RLK_ERR_UNSUPPORTED, std::string(name) + "=" + v +
                                         " is not a planner value the ring protocol model replays");
}

uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d;
    f.s = 0;
    while ((1ull << f.s) < d) ++f.s;
    f.m = (uint32_t)((((uint64_t)1 << 32) * (((uint64_t)1 << f.s) - d)) / d + 1);
    return f;
}

// Whether consumer warps may skip the rows in which they have no tile:
// every warp's first row below first_lim and its consecutive rows at most
// span apart (the tile rotation repeats within NW rows).
//  * Forward (span rbufs, first_lim 2*rbufs).  A warp still waits for the
//    release of row n - rbufs (a parity wait on partfree) before each row it
//    works on, and a parity wait is right only while the barrier is within
//    one phase of it: row n - 2*rbufs must already be released, which the
//    warp's previous wait covered.
//  * L2 fused schedule with skew S (span rbufs - S, first_lim rbufs).  Also
//    a warp in phase B of row n reads rows[b].lse, which the fold of row
//    n + rbufs overwrites.  That fold needs phase A of every row up to
//    n + rbufs in every warp with a tile there (the pushes go in row order);
//    a warp's phase A of rows above n + S comes after its phase B of row n,
//    and rows at most rbufs - S apart put one of them in (n + S, n + rbufs].
//    The first row below rbufs keeps the first lseready parity wait within
//    one phase.
bool row_skip_safe(int NW, int ntl, int span, int first_lim) {
    if (ntl >= NW || span < 1) return false;  // every warp has a tile in every row
    const int step = ntl % NW;
    for (int w = 0; w < NW; ++w) {
        int last = -1, r = 0;
        for (int n = 0; n < 2 * NW + 2 * first_lim; ++n) {
            const int f = ((w - r) % NW + NW) % NW;
            if (f < ntl) {
                if (last < 0 ? n >= first_lim : n - last > span) return false;
                last = n;
            }
            r = (r + step) % NW;
        }
        if (last < 0) return false;
    }
    return true;
}

// Shared-memory layout for NS slots; returns the total bytes.
uint32_t layout(Params& p, int NS) {
    uint32_t off = (uint32_t)NS * (uint32_t)p.slot_bytes;
    p.off_full = off;
    off += 8u * NS;
    p.off_empty = off;
    off += 8u * NS;
    p.off_hdr = align_up(off, 16);
    off = p.off_hdr + (uint32_t)sizeof(SlotHdr) * NS;
    p.off_seq = off;
    off += 4u * NS;
    p.off_part = align_up(off, 16);
    off = p.off_part + (uint32_t)p.rbufs * 8u * (uint32_t)p.NT;
    p.off_fold = off;
    off += 8u * (uint32_t)p.NT;
    p.off_rows = align_up(off, 16);
    off = p.off_rows + (uint32_t)p.rbufs * (uint32_t)sizeof(RowShared);
    p.off_xtin = align_up(off, 16);
    off = p.off_xtin + (uint32_t)p.rbufs * (uint32_t)kMaxCluster * 8u;
    p.off_meta = align_up(off, 16);
    off = p.off_meta + (uint32_t)sizeof(TileMeta) * (uint32_t)((p.NT + p.C - 1) / p.C);
    p.off_tpart = align_up(off, 16);
    if (p.ent) off = p.off_tpart + (uint32_t)p.rbufs * 4u * (uint32_t)p.NT;
    p.off_foldt = align_up(off, 16);
    if (p.ent) off = p.off_foldt + 4u * (uint32_t)p.NT;
    p.off_bars = align_up(off, 8);
    off = p.off_bars + 5u * 8u * (uint32_t)p.rbufs;  // rowdone, lseready, partfree, xbar, lsebar
    p.off_flag = off;
    off += 16u;
    return align_up(off, 128);
}

}  // namespace

rlk_status check_planner_env() {
    int v = 0;
    rlk_status s;
    if ((s = knob("RLK_CTAS_PER_SM", 0, {0, 1, 2}, &v)) != RLK_OK) return s;
    if ((s = knob("RLK_ROW_BUFS", 0, {2, 4, kMaxRowBufs}, &v)) != RLK_OK) return s;
    if ((s = knob("RLK_FUSED_SKEW", -1, {-1, 0, 1, 2, 3, 4, 5, 6, 7}, &v)) != RLK_OK) return s;
    const char* sch = std::getenv("RLK_FUSED_SCHEDULE");
    if (sch && *sch && std::string(sch) != "l2" && std::string(sch) != "resident")
        return fail(RLK_ERR_UNSUPPORTED, "RLK_FUSED_SCHEDULE must be l2 or resident");
    for (const char* gone : {"RLK_TPS", "RLK_MAX_SLOTS", "RLK_LMHEAD_PAIR"}) {
        const char* g = std::getenv(gone);
        if (g && *g) return fail(RLK_ERR_UNSUPPORTED, std::string(gone) + " is not a planner override (unset it)");
    }
    return RLK_OK;
}

rlk_status launch_selftest_wait(uint64_t limit_ns, uint32_t* status, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(e));
    return RLK_OK;
}

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
    p.ent = (a.entropy != nullptr) ? 1 : 0;
    if (p.ent && mode != kModeFwd && mode != kModeFused)
        return fail(RLK_ERR_UNSUPPORTED, "the entropy is computed by the forward and the fused forward+backward");
    // One bulk copy per chunk of tps consecutive tiles, about 8192 columns
    // (16 KB): a copy costs about the same issue time whatever its size, so
    // large copies are what keeps the stream near HBM bandwidth.
    const int tps_target = p.W >= 8192 ? 1 : 8192 / p.W;
    auto set_chunk = [&](int tps) {
        p.tps = tps;
        const int64_t cols = (int64_t)tps * p.W;
        p.slot_bytes = (int32_t)align_up((uint32_t)((((cols + 7) & ~(int64_t)7) + 8) * 2), 16);
    };
    set_chunk(tps_target);
    // The fused schedule: second read from L2 (default) or, with
    // RLK_FUSED_SCHEDULE=resident, the row shard held in shared memory.
    if (mode == kModeFused) {
        const char* sch = std::getenv("RLK_FUSED_SCHEDULE");
        const std::string s = sch ? sch : "";
        if (!s.empty() && s != "l2" && s != "resident")
            return fail(RLK_ERR_UNSUPPORTED, "RLK_FUSED_SCHEDULE must be l2 or resident");
        if (s != "resident") mode = kModeFusedL2;
        if (p.ent && mode != kModeFusedL2)
            return fail(RLK_ERR_UNSUPPORTED, "the entropy is computed by the L2 fused schedule, not the resident one");
        if (a.grpo && mode != kModeFusedL2)
            return fail(RLK_ERR_UNSUPPORTED, "the fused GRPO step runs the L2 fused schedule, not the resident one");
    }
    if (a.grpo && mode != kModeFusedL2) return fail(RLK_ERR_UNSUPPORTED, "the fused GRPO step is a fused mode");
    int C = (mode == kModeBwd) ? 1 : c.virtual_tp;
    // The L2 fused schedule at virtual TP 1 splits each row over a cluster of
    // two CTAs, as the resident schedule does when a row does not fit: every
    // virtual shard is still computed by distinct CTAs and the fold runs in
    // global tile order, so the bits are those of one CTA per row.  With a
    // whole row per CTA the first copies of a row, across the GPU, put about
    // 90 MB between its two reads (some second copies miss L2) and each CTA
    // waits for its own row's fold.
    if (mode == kModeFusedL2 && C == 1 && c.num_tiles % 2 == 0) C = 2;
    // The streaming modes take larger chunks where the CTA's shard allows:
    // the largest number of tiles that divides it and stays within
    // kFusedChunkCols columns (measured: 4 tiles of 2384 columns run 2-7%
    // faster than 3 for kModeFusedL2, which issues twice the copies, and
    // 0.3-1.5% faster for the forward and the backward).  The forward and the
    // backward keep the ~8192-column target where no such divisor reaches
    // half of it (a shard of a prime number of tiles, say).
    if (mode == kModeFusedL2 || mode == kModeFwd || mode == kModeBwd) {
        const int ntl = c.num_tiles / C;
        int best = 1;
        for (int d = 1; d <= ntl; ++d)
            if (ntl % d == 0 && (int64_t)d * p.W <= kFusedChunkCols) best = d;
        if (mode == kModeFusedL2 || 2 * best >= tps_target) set_chunk(best);
    }
    // CTAs per SM.  Two streaming CTAs per SM double the bulk-copy issue rate
    // (two producer warps) and let clusters of 8 cover every SM: measured on
    // GB300 the forward streams at the copy bandwidth with two against 88% of
    // it with one.  The resident fused schedule needs the whole shared
    // memory.  The L2 fused schedule takes two while the rows between a row's
    // two copies, with one row of skew, still fit kL2ReuseBytes at twice the
    // CTAs (virtual TP 4 and 8 at 152576 x 64 tiles); else one while they fit
    // at one CTA per SM (TP 1 and 2); else (nothing fits: a row of an odd
    // number of tiles per CTA, or a very wide one) two with no skew, each CTA
    // covering the other's wait for its row's LSE (measured on GB300 with a
    // whole 152576-column row per CTA: 6.3 ms against 6.6 for one CTA per SM
    // with a row of skew).
    const int64_t shard_bytes = (int64_t)((c.num_tiles + C - 1) / C) * p.W * 2;
    int ctas_per_sm = (mode == kModeFwd || mode == kModeBwd) ? 2 : 1;
    if (mode == kModeFusedL2) {
        const int64_t row1 = shard_bytes * di.sm_count;  // one row shard per SM
        if (kL2ReuseBytes / (2 * row1) >= 2 || kL2ReuseBytes / row1 < 2) ctas_per_sm = 2;
    }
    int forced = 0;
    rlk_status kst = knob("RLK_CTAS_PER_SM", 0, {0, 1, 2}, &forced);
    if (kst != RLK_OK) return kst;
    if (forced == 1 || forced == 2) ctas_per_sm = forced;
    uint32_t budget = (uint32_t)di.smem_optin / (uint32_t)ctas_per_sm - 1024u;
    const int cap = kMaxSlots;
    auto max_slots = [&](Params& q) {
        int lo = 0;
        for (int ns = 1; ns <= cap; ++ns) {
            if (layout(q, ns) <= budget) lo = ns;
            else break;
        }
        return lo;
    };
    // Row buffers of the fold: more buffers let a row's exchange and fold lag
    // further behind phase A (short shards give short rows per CTA); they
    // cost rbufs * (8 * num_tiles + 128) bytes of shared memory.
    {
        // (measured at virtual TP 8: the forward runs 5% faster with 4 than with
        // 8; the fused L2 schedule needs skew + 1 of them)
        const int rb_default = c.num_tiles > 256 ? 2 : (mode == kModeFusedL2 && c.num_tiles <= 128) ? 8 : 4;
        int rb = rb_default;
        if ((kst = knob("RLK_ROW_BUFS", rb_default, {2, 4, kMaxRowBufs}, &rb)) != RLK_OK) return kst;
        if (mode == kModeBwd || mode == kModeFused) rb = 2;
        p.rbufs = rb;
        p.rb_shift = rb == 8 ? 3 : rb == 4 ? 2 : 1;
        // kModeFusedL2 skew: the rows of phase A between a row's two copies
        // must stay in L2.  Keep (skew + 1) rows of every SM's shard within
        // kL2ReuseBytes, skew < rbufs, at most kMaxSkew; at least one row of
        // skew with one CTA per SM (nothing else runs while a CTA waits for its
        // LSE), none needed with two.
        int skew = 1;
        if (mode == kModeFusedL2) {
            const int64_t gpu_row = shard_bytes * di.sm_count * ctas_per_sm;
            int fit = (int)(kL2ReuseBytes / (gpu_row > 0 ? gpu_row : 1));
            skew = fit - 1;
            if (skew > kMaxSkew) skew = kMaxSkew;
            if (skew > rb - 1) skew = rb - 1;
            if (skew < (ctas_per_sm == 2 ? 0 : 1)) skew = ctas_per_sm == 2 ? 0 : 1;
            // skew 0: phase B of a row right after its phase A and LSE
            int forced_skew = -1;
            if ((kst = knob("RLK_FUSED_SKEW", -1, {-1, 0, 1, 2, 3, 4, 5, 6, 7}, &forced_skew)) != RLK_OK) return kst;
            if (forced_skew >= rb)
                return fail(RLK_ERR_UNSUPPORTED, "RLK_FUSED_SKEW must be below the row buffers of the fold");
            if (forced_skew >= 0) skew = forced_skew;
        }
        p.skew = skew;
    }
    int NS = 0;
    p.C = C;
    if (mode == kModeFused) {
        for (;;) {
            p.C = C;
            // Chunks that divide the CTA's tiles evenly pack two rows without waste.
            const int ntl_max = (c.num_tiles + C - 1) / C;
            int tps = tps_target < ntl_max ? tps_target : ntl_max;
            while (tps > 1 && ntl_max % tps) --tps;
            set_chunk(tps);
            NS = max_slots(p);
            // The skewed fused order keeps two rows of this CTA's chunks resident.
            if (NS >= 2 * ((ntl_max + p.tps - 1) / p.tps)) break;
            C *= 2;
            if (C > 8 || C > c.num_tiles)
                return fail(RLK_ERR_UNSUPPORTED,
                            "vocabulary too large to keep a row's shard resident for the single-pass fused "
                            "forward+backward; call rlk_logp_fwd then rlk_logp_bwd with lse_in");
        }
    } else {
        NS = max_slots(p);
        if (NS < kMinSlotsShared && ctas_per_sm == 2 && forced != 2) {
            // wide tiles: one CTA per SM keeps a deeper ring
            ctas_per_sm = 1;
            budget = (uint32_t)di.smem_optin - 1024u;
            NS = max_slots(p);
        }
    }
    if (NS < 1) return fail(RLK_ERR_UNSUPPORTED, "tile too wide for one shared-memory slot");

    const int ntl_cta = (c.num_tiles + p.C - 1) / p.C;
    auto pick = [&](int per_sm) -> void (*)(Params) {
        const bool two = per_sm == 2;
        if (a.grpo) {  // kModeFusedL2 only (checked above)
            if (p.ent)
                return two ? stream_kernel<kModeFusedL2, 2, kFlagGrpo | kFlagEnt>
                           : stream_kernel<kModeFusedL2, 1, kFlagGrpo | kFlagEnt>;
            return two ? stream_kernel<kModeFusedL2, 2, kFlagGrpo> : stream_kernel<kModeFusedL2, 1, kFlagGrpo>;
        }
        if (p.ent && mode == kModeFusedL2)
            return two ? stream_kernel<kModeFusedL2, 2, kFlagEnt> : stream_kernel<kModeFusedL2, 1, kFlagEnt>;
        if (p.ent) return two ? stream_kernel<kModeFwd, 2, kFlagEnt> : stream_kernel<kModeFwd, 1, kFlagEnt>;
        if (two)
            return (mode == kModeFwd)     ? stream_kernel<kModeFwd, 2, 0>
                 : (mode == kModeBwd)     ? stream_kernel<kModeBwd, 2, 0>
                 : (mode == kModeFusedL2) ? stream_kernel<kModeFusedL2, 2, 0>
                                          : stream_kernel<kModeFused, 2, 0>;
        return (mode == kModeFwd)     ? stream_kernel<kModeFwd, 1, 0>
             : (mode == kModeBwd)     ? stream_kernel<kModeBwd, 1, 0>
             : (mode == kModeFusedL2) ? stream_kernel<kModeFusedL2, 1, 0>
                                      : stream_kernel<kModeFused, 1, 0>;
    };
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    cfg.blockDim = dim3(threads_for(mode, ctas_per_sm), 1, 1);
    cfg.stream = stream;
    cfg.numAttrs = 0;
    if (p.C > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)p.C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    // Clusters (or CTAs when C = 1) resident at once for the kernel and
    // shared-memory size; 0 with the message set when none fits.
    auto resident = [&](int per_sm, uint32_t bytes) -> int64_t {
        void (*k)(Params) = pick(per_sm);
        const void* f = reinterpret_cast<const void*>(k);
        cfg.blockDim = dim3(threads_for(mode, per_sm), 1, 1);
        cudaError_t err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (err != cudaSuccess) {
            fail(RLK_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(err));
            return 0;
        }
        cfg.dynamicSmemBytes = bytes;
        if (p.C > 1) {
            cfg.gridDim = dim3((unsigned)(p.C * (di.sm_count / p.C)), 1, 1);
            int n = 0;
            err = cudaOccupancyMaxActiveClusters(&n, k, &cfg);
            if (err != cudaSuccess || n <= 0) {
                fail(RLK_ERR_CUDA, std::string("no cluster of ") + std::to_string(p.C) +
                                       " CTAs fits: " + cudaGetErrorString(err));
                return 0;
            }
            return n;
        }
        int blocks = 0;
        err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, f, (int)cfg.blockDim.x, bytes);
        if (err != cudaSuccess || blocks <= 0) {
            fail(RLK_ERR_CUDA, std::string("kernel does not fit on an SM: ") + cudaGetErrorString(err));
            return 0;
        }
        return (int64_t)blocks * di.sm_count;
    };

    uint32_t smem = layout(p, NS);
    int64_t clusters = resident(ctas_per_sm, smem);
    if (clusters <= 0) return RLK_ERR_CUDA;
    void (*kfn)(Params) = pick(ctas_per_sm);
    cfg.blockDim = dim3(threads_for(mode, ctas_per_sm), 1, 1);
    {
        const int nw = consumers_for(mode, ctas_per_sm);
        p.row_skip = (mode == kModeFwd && row_skip_safe(nw, ntl_cta, p.rbufs, 2 * p.rbufs)) ||
                             (mode == kModeFusedL2 && row_skip_safe(nw, ntl_cta, p.rbufs - p.skew, p.rbufs))
                         ? 1
                         : 0;
    }
    p.NS = NS;
    p.ns_div = make_fastdiv((uint32_t)NS);
    smem = layout(p, NS);
    cfg.dynamicSmemBytes = smem;
    cudaError_t e = cudaSuccess;
    if (clusters > p.T) clusters = p.T;
    {
        // Ring items are numbered in 32 bits per CTA (two blocks of nch
        // chunks per row in the fused schedules); no wrap is allowed.
        const int64_t rows_cta = (p.T + clusters - 1) / clusters;
        const int64_t nch_cta = (ntl_cta + p.tps - 1) / p.tps;
        if (rows_cta * 2 * nch_cta >= ((int64_t)1 << 31))
            return fail(RLK_ERR_UNSUPPORTED, "too many rows per CTA for the slot ring's 32-bit item numbers");
    }
    cfg.gridDim = dim3((unsigned)(clusters * p.C), 1, 1);
    if (env_int("RLK_VERBOSE", 0))
        std::fprintf(stderr,
                     "rlk stream plan: mode %d, %d CTA(s)/SM, %lld clusters x %d CTAs, %d tiles/copy, %d slots of %d B, "
                     "%d row buffers, skew %d, row skip %d, %u B shared memory, %d consumer warps\n",
                     mode, ctas_per_sm, (long long)clusters, p.C, p.tps, p.NS, p.slot_bytes, p.rbufs, p.skew,
                     p.row_skip, smem, consumers_for(mode, ctas_per_sm));
    e = cudaLaunchKernelEx(&cfg, kfn, p);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(e));
    return RLK_OK;
}

}  // namespace rlk
