// Fused lm_head variant (sm_103a): the selected-token log-probability of
// logits = hidden @ W^T without materialising the logits, and its gradients
// with respect to hidden and W.
//
// The optional fused kernel of issue #323 ("[WS2][Logprob] H100 validation
// and reproduction guide", "Validation Boundary": "the optional PR6 fused
// kernel") is the prior art; its design is not on the pages.  Here each
// (128-token block, 256-row chunk of a global vocabulary tile) unit runs a
// tcgen05 GEMM (accumulators in tensor memory, operands staged by TMA with
// the 128-byte swizzle), and the epilogue turns the chunk into its (max,
// sumexp) partial -- of FP32 logits that are never rounded or written.  A
// fold kernel merges each tile's chunks in chunk order into the tile's
// partial, then the tiles in fixed index order (rlk_fold.cuh), and forms
// logp.
//
// Roles (192 threads, one CTA per SM): warp 0 issues the TMA loads, warp 1
// allocates tensor memory and issues the MMAs, warps 2-5 run the epilogue
// (warp w reads TMEM lanes 32*(w%4)..+31, one token row per thread).
// Units are handed out by an atomic ticket in chunk-major order within bands
// of token blocks: the units in flight at any moment are a window of
// consecutive units, so the token blocks that share a weight chunk run
// together and the weight is read from HBM once per band.  The producer's
// lane takes the ticket and passes the unit to the other roles through a
// small queue in shared memory.
// Virtual TP: the CTAs are split into virtual_tp groups; group j takes
// tickets only for the tiles of shard j.  A chunk's partial is computed by
// one thread in one fixed order (32-column blocks, then columns) and a tile's
// chunks are merged in chunk order, whatever the grouping or the CTA that
// runs them, so outputs do not depend on virtual_tp.
//
// Backward: dlogits = g (onehot - exp(x - LSE)) in BF16.  In the forward +
// backward call the forward also stores its FP32 logits (each epilogue warp
// stages 32 rows x 32 columns in shared memory with the 128-byte swizzle and
// issues one TMA tile store) and an elementwise pass forms dlogits once the
// fold has the LSE; the backward from
// a given LSE re-runs the GEMM with an epilogue that writes dlogits.  The
// logits are the same accumulators either way, so dlogits are bitwise equal.
// Then one persistent launch runs the two gradient contractions as tcgen05
// GEMMs with FP32 accumulators:
//   dHidden[T, H]  = dlogits[:, :V_real] W[:V_real]      (A K-major, B MN-major)
//   dW[V_padded, H] = dlogits[:, :V_real]^T hidden       (A and B MN-major)
// Each output tile accumulates its whole K range in one fixed order on one
// CTA: no split-K, no atomics on data.  An MN-major B operand (W, hidden)
// arrives as four 64-wide swizzled blocks per stage in one 3-D TMA box
// (make_map_mn3): four 2-D boxes a stage measured latency-bound.
//
// Every wait is bounded; on expiry the CTA records RLK_ERR_TIMEOUT, stops
// issuing, waits (bounded) for its issued copies and MMAs, frees its tensor
// memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>
#include <string>

#include "rlk_fold.cuh"
#include "rlk_internal.h"
#include "rlk_ptx.cuh"

namespace rlk {
namespace {

// TMA tile store from shared memory (bulk group); the writing threads fence
// the async proxy first.
__device__ __forceinline__ void tma_store_2d(const void* tmap, int32_t c0, int32_t c1, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(tmap), "r"(c0),
                 "r"(c1), "r"(src)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The source of every committed store has been read (the buffer may be rewritten).
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Every committed store has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

constexpr int kBM = 128;  // token rows per unit (TMEM lanes)
constexpr int kBN = 256;  // vocabulary rows per chunk (accumulator columns)
constexpr int kBK = 64;   // K per stage: 64 BF16 = one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kUq = 4;  // depth of the unit queue from the producer to the other roles
constexpr int kThreadsLm = 192;
constexpr uint32_t kTmemCols = 512;  // two accumulators of kBN columns
constexpr uint32_t kStageA = kBM * kBK * 2;
constexpr uint32_t kStageB = kBN * kBK * 2;
constexpr uint32_t kMnBlock = 64 * kBK * 2;  // one 64-wide block of an MN-major stage: 64 K rows x 128 B
constexpr uint64_t kDrainNsLm = 1000000000ull;
constexpr int kMaxGroups = 8;
// Unit order of the logits GEMMs: a unit is one 256-row weight chunk of one token block; units
// come in bands of token blocks whose hidden spans at most kBandHiddenBytes, chunk-major within a
// band, hidden loaded with an L2 evict-last policy.  The units in flight then share about two
// weight chunks (a few MB) and one band of hidden, so L2 holds both and the weight is read from
// HBM once per band.  Measured at 8192 x 4096 x 152576 (time, DRAM reads of the forward GEMM):
// bands of 64 MB 6.43 ms, 13.9 GB (hidden no longer stays in L2); 32 MB 5.77 ms, 2.57 GB (the
// weight twice); 16 MB 6.06 ms; an evict-first hint on the weight loads made every band size
// slower (64 MB 6.25 ms, 10.3 GB; 32 MB 5.92 ms).  Whole-tile units in bands of 32 blocks had
// measured 5.88 ms and 3.75 GB: the ten chunks of a tile ran on one CTA, so the units in flight
// spanned about 47 MB of weight.
constexpr int64_t kBandHiddenBytes = (int64_t)32 << 20;
constexpr int kKeepHidden = 1;   // 1: the logits GEMMs load hidden with an L2 evict-last policy
// Tile order of the gradient GEMMs: bands of kBandN 256-wide H blocks, M-major within a band.
// Measured at 8192 x 4096 x 152576 (DRAM reads, time of the gradient launch): bands of 16 (no
// banding at H = 4096) 26.1 GB, 14.12 ms; of 8 16.6 GB, 13.89 ms; of 4 23.5 GB, 13.92 ms.  An L2
// evict-last hint on dW's hidden loads did not help (16.8 GB at bands of 8).
constexpr int kBandN = 8;
// Workspace: 256 bytes of tickets (three launches x kMaxGroups 64-bit counters).
constexpr size_t kTicketBytes = 256;

// kEpiPartials: chunk partials and target logits; kEpiPartialsStore: the same,
// and the FP32 logits written to a [T, V_padded] buffer; kEpiGrad: dlogits.
enum : int { kEpiPartials = 0, kEpiGrad = 1, kEpiPartialsStore = 2 };

struct Bars {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t ufull[kUq];   // unit queue entry written (the producer's arrival)
    uint64_t uempty[kUq];  // entry read by the MMA thread and the four epilogue warps
    uint64_t drain;
    int64_t unit[kUq];
    uint32_t tmem_addr;
    int abort_flag;
};

// Shared memory of the logits GEMMs past the 1024-byte alignment slack: the
// operand stages, then the barriers (then, for kEpiPartialsStore, the staging
// blocks of the logits store).
constexpr size_t kGemmSmemCore = ((size_t)kStages * (kStageA + kStageB) + sizeof(Bars) + 1023) / 1024 * 1024;
// Per epilogue warp: 32 rows x 32 FP32 columns with the 128-byte swizzle (the
// TMA store's source), or 32 rows at pitch 33 (the 16-column remainder).
constexpr int kStoreStage = 1280;  // floats (5 KB, a multiple of 1024 bytes)

struct WaitCtl {
    uint32_t* status;
    uint64_t wait_ns;
};

__device__ bool lm_wait(Bars* bars, uint32_t bar, uint32_t parity, const WaitCtl& w) {
    if (mbar_try_wait(bar, parity)) return true;
    volatile int* ab = &bars->abort_flag;
    if (*ab) return false;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*ab) return false;
        if (globaltimer_ns() - t0 > w.wait_ns) {
            *ab = 1;
            atomicOr(w.status, kStatusTimeout);
            return false;
        }
    }
}

__device__ void lm_drain_wait(uint32_t bar, uint32_t parity, const WaitCtl& w) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kDrainNsLm) {
            atomicOr(w.status, kStatusTimeout);
            return;
        }
    }
}

// The producer publishes the CTA's n-th unit (-1: no more units).
__device__ bool unit_put(Bars* bars, int64_t n, int64_t u, const WaitCtl& w) {
    const int s = (int)(n % kUq);
    const uint32_t par = (uint32_t)((n / kUq) & 1);
    if (!lm_wait(bars, smem_u32(&bars->uempty[s]), par ^ 1u, w)) return false;
    *reinterpret_cast<volatile int64_t*>(&bars->unit[s]) = u;
    mbar_arrive(smem_u32(&bars->ufull[s]));  // release: the entry is visible to whoever acquires the phase
    return true;
}

__device__ bool unit_get(Bars* bars, int64_t n, int64_t& u, const WaitCtl& w) {
    const int s = (int)(n % kUq);
    if (!lm_wait(bars, smem_u32(&bars->ufull[s]), (uint32_t)((n / kUq) & 1), w)) return false;
    u = *reinterpret_cast<volatile int64_t*>(&bars->unit[s]);
    return true;
}

__device__ __forceinline__ void unit_done(Bars* bars, int64_t n) { mbar_arrive(smem_u32(&bars->uempty[n % kUq])); }

__device__ void init_bars(Bars* bars) {
    for (int s = 0; s < kStages; ++s) {
        mbar_init(smem_u32(&bars->full[s]), 1);
        mbar_init(smem_u32(&bars->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
        mbar_init(smem_u32(&bars->tfull[b]), 1);
        mbar_init(smem_u32(&bars->tempty[b]), 4);
    }
    for (int s = 0; s < kUq; ++s) {
        mbar_init(smem_u32(&bars->ufull[s]), 1);
        mbar_init(smem_u32(&bars->uempty[s]), 5);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort_flag = 0;
    fence_mbar_init();
}

// The producer's final step: every copy it issued lands before the CTA may exit.
__device__ void drain_copies(Bars* bars, int64_t issued, const WaitCtl& w) {
    const int64_t first = issued > kStages ? issued - kStages : 0;
    for (int64_t j = first; j < issued; ++j)
        lm_drain_wait(smem_u32(&bars->full[j % kStages]), (uint32_t)((j / kStages) & 1), w);
}

// ----------------------------------------------------------------- logits GEMM (forward partials / dlogits)

struct LmParams {
    const int64_t* targets;
    const uint8_t* mask;
    float2* partials;  // [T, NT * nchunk] chunk partials (kEpiPartials)
    float* xt;         // [T] target logits          (kEpiPartials)
    float* xlog;       // [T, Vp] FP32 logits out     (kEpiPartialsStore)
    const float* lse_in;  // [T]                      (kEpiGrad)
    const float* grad;    // [T] upstream g of logp   (kEpiGrad)
    uint16_t* dlogits;    // [T, Vp] BF16 out         (kEpiGrad)
    unsigned long long* tickets;  // one per virtual-TP group, 0 at launch
    WaitCtl w;
    int64_t T, Vr, Vp, ignore_index;
    int32_t K, NT, W, vtp, nchunk, rem, mask_mode;
    int32_t MB;   // token blocks
    int32_t MBg;  // token blocks per band of the unit order (unit_coords)
    int32_t keep_hidden;  // hidden tiles loaded with an L2 evict-last policy
};

// Virtual-TP group of this CTA: group j takes tickets for the units
// [0, NT/vtp * nchunk * MB) of shard j (unit_coords).
struct Group {
    int j, tile0, ntl;
    int64_t end;
};

__device__ Group group_of(const LmParams& p) {
    const int Gj = (int)gridDim.x / p.vtp;
    Group g;
    g.j = (int)blockIdx.x / Gj;
    g.ntl = p.NT / p.vtp;
    g.tile0 = g.j * g.ntl;
    g.end = (int64_t)g.ntl * p.nchunk * p.MB;
    return g;
}

// Unit u of a group is (weight chunk ch of tile, token block mb).  Token
// blocks are taken in bands of p.MBg blocks; within a band the order is
// chunk-major over the shard's tiles, so the units in flight share about two
// weight chunks (the band's blocks of one chunk run together) and one band of
// hidden.  The last band may be narrower.
__device__ __forceinline__ void unit_coords(const LmParams& p, const Group& g, int64_t u, int& tile, int& ch,
                                            int& mb) {
    const int64_t band_units = (int64_t)g.ntl * p.nchunk * p.MBg;
    const int64_t full = p.MB / p.MBg;
    int64_t gc;
    if (u < full * band_units) {
        const int64_t b = u / band_units, r = u % band_units;
        gc = r / p.MBg;
        mb = (int)(b * p.MBg + r % p.MBg);
    } else {
        const int64_t r = u - full * band_units;
        const int w = p.MB - (int)full * p.MBg;
        gc = r / w;
        mb = (int)(full * p.MBg + r % w);
    }
    tile = g.tile0 + (int)(gc / p.nchunk);
    ch = (int)(gc % p.nchunk);
}

// One 32-column block of a row's logits into the running partial of its
// tile: exact block max, rescale when it grows, then the block's sum of
// exp(x - m) with four accumulators added in a fixed order.
__device__ __forceinline__ void online_block(const float (&v)[32], int nv, int64_t col0, int64_t Vr, float& m_run,
                                             float& s_run) {
    float bm = -INFINITY;
#pragma unroll
    for (int i = 0; i < 32; ++i)
        if (i < nv && col0 + i < Vr) bm = fmax_nan(bm, v[i]);
    if (bm > m_run || bm != bm) {
        s_run = __fmul_rn(s_run, ex2_approx(__fmul_rn(__fsub_rn(m_run, bm), kLog2e)));
        m_run = bm;
    }
    if (m_run == -INFINITY) return;  // nothing finite yet: the identity
    const float nmL = -__fmul_rn(m_run, kLog2e);
    float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        const bool ok = i < nv && col0 + i < Vr;
        const float e = ok ? ex2_approx(__fmaf_rn(v[i], kLog2e, nmL)) : 0.f;
        a[i & 3] = __fadd_rn(a[i & 3], e);
    }
    s_run = __fadd_rn(s_run, __fadd_rn(__fadd_rn(a[0], a[1]), __fadd_rn(a[2], a[3])));
}

// dlogits of one 32-column block of a row: g * ([c == t] - exp(x - LSE)) on
// real columns of an active row, exactly 0 elsewhere; BF16, stored as
// nv / 8 16-byte vectors (nv is 32 or 16).
__device__ __forceinline__ void grad_block(const float (&v)[32], int nv, int64_t col0, int64_t Vr, bool active,
                                           int64_t target, float g, float nlL, uint16_t* drow) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        float d[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const int64_t c = col0 + i + j;
            float dj = 0.f;
            if (active && c < Vr && i + j < nv) {
                const float pr = ex2_approx(__fmaf_rn(v[i + j], kLog2e, nlL));
                dj = (c == target) ? __fmul_rn(g, __fsub_rn(1.f, pr)) : __fmul_rn(-g, pr);
            }
            d[j] = dj;
        }
        w[i >> 1] = pack_bf16x2_rn(d[0], d[1]);
    }
    uint4* out = reinterpret_cast<uint4*>(drow + col0);
#pragma unroll
    for (int q = 0; q < 4; ++q)
        if (q * 8 < nv) out[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
}

template <int EPI>
__global__ void __launch_bounds__(kThreadsLm, 1)
    lmhead_kernel(const __grid_constant__ CUtensorMap tmH, const __grid_constant__ CUtensorMap tmW,
                  const __grid_constant__ CUtensorMap tmWr, const __grid_constant__ CUtensorMap tmX,
                  const __grid_constant__ LmParams p) {
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte alignment for the 128-byte-swizzled operand tiles.
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* sA = smem;
    unsigned char* sB = smem + kStages * kStageA;
    Bars* bars = reinterpret_cast<Bars*>(smem + kStages * (kStageA + kStageB));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = p.K / kBK;

    if (threadIdx.x == 0) init_bars(bars);
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_addr), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_addr;
    const Group grp = group_of(p);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0, n = 0;
            bool aborted = false;
            const uint64_t keep = l2_policy_evict_last();
            while (!aborted) {
                int64_t u = (int64_t)atomicAdd(&p.tickets[grp.j], 1ull);
                if (u >= grp.end) u = -1;
                if (!unit_put(bars, n++, u, p.w) || u < 0) break;
                int tile, ch, mb;
                unit_coords(p, grp, u, tile, ch, mb);
                const bool last_rem = (ch == p.nchunk - 1) && p.rem;
                const int nrows = last_rem ? p.rem : kBN;
                const int n0 = tile * p.W + ch * kBN;
                for (int kb = 0; kb < KB; ++kb) {
                    if (!lm_wait(bars, smem_u32(&bars->empty[stage]), phase ^ 1u, p.w)) {
                        aborted = true;
                        break;
                    }
                    const uint32_t fb = smem_u32(&bars->full[stage]);
                    mbar_arrive_expect_tx(fb, kStageA + (uint32_t)nrows * kBK * 2);
                    if (p.keep_hidden)
                        tma_load_2d_hint(smem_u32(sA + stage * kStageA), &tmH, kb * kBK, mb * kBM, fb, keep);
                    else
                        tma_load_2d(smem_u32(sA + stage * kStageA), &tmH, kb * kBK, mb * kBM, fb);
                    tma_load_2d(smem_u32(sB + stage * kStageB), last_rem ? &tmWr : &tmW, kb * kBK, n0, fb);
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            drain_copies(bars, issued, p.w);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t chunk = 0, n = 0;
            bool aborted = false;
            while (!aborted) {
                int64_t u;
                if (!unit_get(bars, n, u, p.w)) break;
                unit_done(bars, n++);
                if (u < 0) break;
                int tile, ch, mb;
                unit_coords(p, grp, u, tile, ch, mb);
                const int acc = (int)(chunk & 1);
                const uint32_t accph = (uint32_t)((chunk >> 1) & 1);
                ++chunk;
                if (!lm_wait(bars, smem_u32(&bars->tempty[acc]), accph ^ 1u, p.w)) break;
                tc_fence_after();
                const bool last_rem = (ch == p.nchunk - 1) && p.rem;
                const uint32_t idesc = idesc_bf16_f32(kBM, last_rem ? (uint32_t)p.rem : (uint32_t)kBN);
                const uint32_t d = tmem + (uint32_t)(acc * kBN);
                for (int kb = 0; kb < KB; ++kb) {
                    if (!lm_wait(bars, smem_u32(&bars->full[stage]), phase, p.w)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * kStageA);
                    const uint32_t b0 = smem_u32(sB + stage * kStageB);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk)
                        umma_bf16(d, smem_desc_sw128(a0 + kk * 32), smem_desc_sw128(b0 + kk * 32), idesc,
                                  (kb | kk) != 0);
                    umma_commit(smem_u32(&bars->empty[stage]));  // frees the stage when these MMAs finish
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!aborted) umma_commit(smem_u32(&bars->tfull[acc]));
            }
            // Every issued MMA completes before tensor memory is freed.
            umma_commit(smem_u32(&bars->drain));
            lm_drain_wait(smem_u32(&bars->drain), 0u, p.w);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int quarter = warp & 3;
        const int r_in = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        float* xst = reinterpret_cast<float*>(smem + kGemmSmemCore) + quarter * kStoreStage;
        bool store_pending = false;
        int64_t chunk = 0, n = 0;
        for (;;) {
            int64_t u = -1;
            const bool got = unit_get(bars, n, u, p.w);
            if (!__all_sync(0xFFFFFFFFu, got)) break;
            __syncwarp();
            if (lane == 0) unit_done(bars, n);
            ++n;
            if (u < 0) break;
            int tile, ch, mb;
            unit_coords(p, grp, u, tile, ch, mb);
            const int64_t row = (int64_t)mb * kBM + r_in;
            const bool valid = row < p.T;
            int64_t target = -1;
            bool active = false;
            if (valid) {
                target = p.targets[row];
                active = (p.mask_mode == RLK_MASK_EXPLICIT) ? (p.mask[row] != 0) : (target != p.ignore_index);
            }
            float m_run = -INFINITY, s_run = 0.f, xt = 0.f;
            bool have_xt = false;
            float g = 0.f, nlL = 0.f;
            uint16_t* drow = nullptr;
            if (EPI == kEpiGrad && valid) {
                g = p.grad[row];
                const float l = p.lse_in[row];
                nlL = -__fmul_rn(l, kLog2e);
                drow = p.dlogits + row * p.Vp;
                // the device conditions of a backward given the LSE, reported once per row
                if (active && tile == grp.tile0 && ch == 0 && grp.j == 0) {
                    if (target < 0 || target >= p.Vr) atomicOr(p.w.status, kStatusTargetRange);
                    if (!isfinite(l)) atomicOr(p.w.status, kStatusNonFinite);
                }
            }
            const int acc = (int)(chunk & 1);
            const uint32_t accph = (uint32_t)((chunk >> 1) & 1);
            ++chunk;
            const bool ok = lm_wait(bars, smem_u32(&bars->tfull[acc]), accph, p.w);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            const int ncols = ((ch == p.nchunk - 1) && p.rem) ? p.rem : kBN;
            const int64_t cbase = (int64_t)tile * p.W + (int64_t)ch * kBN;
            for (int sub = 0; sub * 32 < ncols; ++sub) {
                float v[32];
                tmem_ld32(tmem + lane_base + (uint32_t)(acc * kBN + sub * 32), v);
                const int nv = min(32, ncols - sub * 32);
                const int64_t col0 = cbase + sub * 32;
                if (EPI == kEpiGrad) {
                    if (valid) grad_block(v, nv, col0, p.Vr, active, target, g, nlL, drow);
                    continue;
                }
                if (EPI == kEpiPartialsStore) {
                    const int64_t row0 = (int64_t)mb * kBM + quarter * 32;
                    // the warp's previous TMA store has read the staging block
                    if (store_pending) {
                        if (lane == 0) bulk_wait_read_all();
                        __syncwarp();
                    }
                    if (nv == 32) {
                        // 32 rows x 128 bytes with the 128-byte swizzle (16-byte chunk j of row r
                        // at chunk j ^ (r mod 8)), then one TMA tile store; rows past T are clipped
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            *reinterpret_cast<float4*>(xst + lane * 32 + ((j ^ (lane & 7)) * 4)) =
                                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(&tmX, (int32_t)col0, (int32_t)row0, smem_u32(xst));
                            bulk_commit();
                        }
                        store_pending = true;
                    } else {
                        // a 16-column remainder: through shared memory at pitch 33 (conflict-free
                        // both ways), then one 64-byte row segment per store
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (i < nv) xst[lane * 33 + i] = v[i];
                        __syncwarp();
                        for (int rr = 0; rr < 32; ++rr)
                            if (row0 + rr < p.T && lane < nv)
                                p.xlog[(row0 + rr) * p.Vp + col0 + lane] = xst[rr * 33 + lane];
                        __syncwarp();
                        store_pending = false;
                    }
                }
                online_block(v, nv, col0, p.Vr, m_run, s_run);
                if (active && target >= col0 && target < col0 + nv && target < p.Vr) {
                    const int idx = (int)(target - col0);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i == idx) xt = v[i];
                    have_xt = true;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->tempty[acc]));
            if (EPI != kEpiGrad && valid) {
                const int64_t k = (int64_t)tile * p.nchunk + ch;
                p.partials[row * (int64_t)p.NT * p.nchunk + k] = make_float2(m_run, s_run);
                if (have_xt) p.xt[row] = xt;
            }
        }
        // the warp's TMA stores complete before the CTA exits
        if (EPI == kEpiPartialsStore && lane == 0) bulk_wait_all();
        __syncwarp();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// A tile's partial from its chunk partials, merged in chunk order: the
// running maximum, the sum rescaled when the maximum grows, then the chunk's
// sum scaled to it.  An all -inf chunk is the identity; a NaN maximum stays.
__device__ __forceinline__ float2 merge_chunks(const float2* c, int nchunk) {
    float m = -INFINITY, s = 0.f;
    for (int k = 0; k < nchunk; ++k) {
        const float2 q = c[k];
        if (q.x == -INFINITY) continue;
        const float M = fmax_nan(m, q.x);
        if (M != m) s = __fmul_rn(s, ex2_approx(__fmul_rn(__fsub_rn(m, M), kLog2e)));
        s = __fadd_rn(s, __fmul_rn(q.y, ex2_approx(__fmul_rn(__fsub_rn(q.x, M), kLog2e))));
        m = M;
    }
    return make_float2(m, s);
}

// LSE and logp of each row from its chunk partials (one warp per row): each
// lane merges the chunks of its tiles, then the tiles are folded in index
// order as in the streaming path.
__global__ void lmhead_fold_kernel(const float2* partials, const float* xt, const int64_t* targets,
                                   const uint8_t* mask, int mask_mode, int64_t ignore_index, int64_t T, int64_t Vr,
                                   int NT, int nchunk, float* logp, float* lse, uint32_t* status) {
    extern __shared__ float2 scratch[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    float2* sc = scratch + (size_t)warp * NT;
    for (int64_t row = (int64_t)blockIdx.x * wpb + warp; row < T; row += (int64_t)gridDim.x * wpb) {
        const float2* pr = partials + row * (int64_t)NT * nchunk;
        for (int t = lane; t < NT; t += 32) sc[t] = merge_chunks(pr + (int64_t)t * nchunk, nchunk);
        __syncwarp();
        // fold_tiles reads each tile's entry before it writes that index of its scratch, so the
        // merged tiles may serve as both
        const float l = fold_tiles(sc, NT, sc, lane);
        if (lane == 0) {
            const int64_t t = targets[row];
            const bool active = (mask_mode == RLK_MASK_EXPLICIT) ? (mask[row] != 0) : (t != ignore_index);
            lse[row] = l;
            if (!active) {
                logp[row] = 0.f;
            } else if (t < 0 || t >= Vr) {
                logp[row] = __int_as_float(0x7FC00000);
                atomicOr(status, kStatusTargetRange);
            } else {
                logp[row] = __fsub_rn(xt[row], l);
            }
            if (active && !isfinite(l)) atomicOr(status, kStatusNonFinite);
        }
        __syncwarp();
    }
}

// dlogits from the FP32 logits the forward stored: g * ([c == t] - exp(x - LSE))
// on the real columns of an active row, exactly 0 elsewhere, BF16 -- the
// operations of grad_block on the same FP32 values, so the result is bitwise
// that of the recompute GEMM's epilogue.  One CTA a row (a grid-stride loop
// past 2^31 - 1 rows), 8 columns (two 16-byte loads, one 16-byte store) a
// thread per step; both streams are read or written once, with the
// cache-streaming hint.
__global__ void __launch_bounds__(256) lmhead_dlogits_kernel(const float* xlog, const float* lse,
                                                             const float* grad, const int64_t* targets,
                                                             const uint8_t* mask, int mask_mode,
                                                             int64_t ignore_index, int64_t T, int64_t Vr,
                                                             int64_t Vp, uint16_t* dlogits, uint32_t* status) {
    const int64_t groups = Vp / 8;
    for (int64_t row = blockIdx.x; row < T; row += gridDim.x) {
        const int64_t t = targets[row];
        const bool active = (mask_mode == RLK_MASK_EXPLICIT) ? (mask[row] != 0) : (t != ignore_index);
        const float g = grad[row];
        const float l = lse[row];
        const float nlL = -__fmul_rn(l, kLog2e);
        // the device conditions of a backward given the LSE, once per row (the target is
        // only compared with column indices, never used as one)
        if (threadIdx.x == 0 && active) {
            if (t < 0 || t >= Vr) atomicOr(status, kStatusTargetRange);
            if (!isfinite(l)) atomicOr(status, kStatusNonFinite);
        }
        const float4* xr = reinterpret_cast<const float4*>(xlog + row * Vp);
        uint4* dr = reinterpret_cast<uint4*>(dlogits + row * Vp);
        for (int64_t q = threadIdx.x; q < groups; q += blockDim.x) {
            const int64_t c0 = q * 8;
            uint4 o = make_uint4(0u, 0u, 0u, 0u);
            if (active && c0 < Vr) {
                const float4 a = __ldcs(&xr[2 * q]), b = __ldcs(&xr[2 * q + 1]);
                const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
                uint32_t w[4];
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    float d[2];
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int64_t c = c0 + i + j;
                        float dj = 0.f;
                        if (c < Vr) {
                            const float pr = ex2_approx(__fmaf_rn(x[i + j], kLog2e, nlL));
                            dj = (c == t) ? __fmul_rn(g, __fsub_rn(1.f, pr)) : __fmul_rn(-g, pr);
                        }
                        d[j] = dj;
                    }
                    w[i >> 1] = pack_bf16x2_rn(d[0], d[1]);
                }
                o = make_uint4(w[0], w[1], w[2], w[3]);
            }
            __stcs(&dr[q], o);
        }
    }
}

// ----------------------------------------------------------------- gradient GEMMs (dHidden and dW)

// Two problems share one persistent launch and one ticket: tiles [0, n0) of
// problem 0 (dHidden, M = T, K = V_real) come first, then tiles [n0, n0 + n1)
// of problem 1 (dW, M = V_padded, K = T); both have N = H in blocks of 256
// (the last one possibly narrower, in 64-wide steps) and a 128-row M block.
// The long dHidden tiles go first so that the short dW tiles fill the tail.
struct GradParams {
    uint16_t* dhidden;  // [T, H] BF16
    uint16_t* dw_bf16;  // [V_padded, H] BF16, or NULL
    float* dw_f32;      // [V_padded, H] FP32, or NULL
    unsigned long long* ticket;
    WaitCtl w;
    int64_t T, Vr, Vp, n0, n1;
    int32_t H, NB, KB0, KB1;  // n-blocks of H; K blocks of problem 0 (V_real) and problem 1 (T)
    int32_t NBg;              // H blocks per band of the tile order (grad_tile)
};

struct GradTile {
    int prob;  // 0: dHidden, 1: dW
    int64_t mb;
    int nb, nbox, KB;
};

__device__ __forceinline__ GradTile grad_tile(const GradParams& p, int64_t u) {
    GradTile t;
    t.prob = u < p.n0 ? 0 : 1;
    const int64_t v = t.prob ? u - p.n0 : u;
    // bands of p.NBg H blocks: M-major within a band (the band's H blocks of one M block run together)
    const int64_t MBp = (t.prob ? p.n1 : p.n0) / p.NB;
    const int64_t band_tiles = MBp * p.NBg;
    const int64_t full = p.NB / p.NBg;
    if (v < full * band_tiles) {
        const int64_t b = v / band_tiles, r = v % band_tiles;
        t.mb = r / p.NBg;
        t.nb = (int)(b * p.NBg + r % p.NBg);
    } else {
        const int64_t r = v - full * band_tiles;
        const int w = p.NB - (int)full * p.NBg;
        t.mb = r / w;
        t.nb = (int)(full * p.NBg + r % w);
    }
    const int left = p.H - t.nb * kBN;
    t.nbox = left >= kBN ? 4 : left / 64;
    t.KB = t.prob ? p.KB1 : p.KB0;
    return t;
}

__global__ void __launch_bounds__(kThreadsLm, 1)
    lmhead_grad_kernel(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmB0,
                       const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                       const __grid_constant__ GradParams p) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem =
        reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* sA = smem;
    unsigned char* sB = smem + kStages * kStageA;
    Bars* bars = reinterpret_cast<Bars*>(smem + kStages * (kStageA + kStageB));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t total = p.n0 + p.n1;

    if (threadIdx.x == 0) init_bars(bars);
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_addr), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_addr;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0, n = 0;
            bool aborted = false;
            while (!aborted) {
                int64_t u = (int64_t)atomicAdd(p.ticket, 1ull);
                if (u >= total) u = -1;
                if (!unit_put(bars, n++, u, p.w) || u < 0) break;
                const GradTile t = grad_tile(p, u);
                const int m0 = (int)(t.mb * kBM);
                const int h0 = t.nb * kBN;
                for (int kb = 0; kb < t.KB; ++kb) {
                    if (!lm_wait(bars, smem_u32(&bars->empty[stage]), phase ^ 1u, p.w)) {
                        aborted = true;
                        break;
                    }
                    const uint32_t fb = smem_u32(&bars->full[stage]);
                    const uint32_t a = smem_u32(sA + stage * kStageA);
                    const uint32_t b = smem_u32(sB + stage * kStageB);
                    // B: the four 64-wide blocks of the stage in one 3-D box (blocks past H read as
                    // zero and still count their bytes)
                    mbar_arrive_expect_tx(fb, kStageA + 4u * kMnBlock);
                    if (t.prob == 0) {
                        // dlogits rows m0.., columns (K) kb*64..; W rows (K) kb*64.., columns h
                        tma_load_2d(a, &tmA0, kb * kBK, m0, fb);
                        tma_load_3d(b, &tmB0, 0, kb * kBK, h0 / 64, fb);
                    } else {
                        // dlogits columns (M) m0.., rows (K) kb*64..; hidden rows (K) kb*64.., columns h
                        tma_load_2d(a, &tmA1, m0, kb * kBK, fb);
                        tma_load_2d(a + kMnBlock, &tmA1, m0 + 64, kb * kBK, fb);
                        tma_load_3d(b, &tmB1, 0, kb * kBK, h0 / 64, fb);
                    }
                    ++issued;
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            drain_copies(bars, issued, p.w);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t tiles = 0, n = 0;
            bool aborted = false;
            while (!aborted) {
                int64_t u;
                if (!unit_get(bars, n, u, p.w)) break;
                unit_done(bars, n++);
                if (u < 0) break;
                const GradTile t = grad_tile(p, u);
                const int acc = (int)(tiles & 1);
                const uint32_t accph = (uint32_t)((tiles >> 1) & 1);
                ++tiles;
                if (!lm_wait(bars, smem_u32(&bars->tempty[acc]), accph ^ 1u, p.w)) break;
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32_major(kBM, (uint32_t)(64 * t.nbox), t.prob == 1, true);
                const uint32_t d = tmem + (uint32_t)(acc * kBN);
                for (int kb = 0; kb < t.KB; ++kb) {
                    if (!lm_wait(bars, smem_u32(&bars->full[stage]), phase, p.w)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = smem_u32(sA + stage * kStageA);
                    const uint32_t b0 = smem_u32(sB + stage * kStageB);
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        // K-major A advances 16 elements (32 B) within its swizzle rows; an
                        // MN-major operand advances two 8-row K groups (2 x 1024 B).
                        const uint64_t ad = t.prob == 0 ? smem_desc_sw128(a0 + kk * 32)
                                                        : smem_desc_sw128_mn(a0 + kk * 2048, kMnBlock, 1024);
                        const uint64_t bd = smem_desc_sw128_mn(b0 + kk * 2048, kMnBlock, 1024);
                        umma_bf16(d, ad, bd, idesc, (kb | kk) != 0);
                    }
                    umma_commit(smem_u32(&bars->empty[stage]));
                    if (++stage == kStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!aborted) umma_commit(smem_u32(&bars->tfull[acc]));
            }
            umma_commit(smem_u32(&bars->drain));
            lm_drain_wait(smem_u32(&bars->drain), 0u, p.w);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5): TMEM -> BF16 / FP32 rows
        const int quarter = warp & 3;
        const int r_in = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        int64_t tiles = 0, n = 0;
        for (;;) {
            int64_t u = -1;
            const bool got = unit_get(bars, n, u, p.w);
            if (!__all_sync(0xFFFFFFFFu, got)) break;
            __syncwarp();
            if (lane == 0) unit_done(bars, n);
            ++n;
            if (u < 0) break;
            const GradTile t = grad_tile(p, u);
            const int acc = (int)(tiles & 1);
            const uint32_t accph = (uint32_t)((tiles >> 1) & 1);
            ++tiles;
            const bool ok = lm_wait(bars, smem_u32(&bars->tfull[acc]), accph, p.w);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;
            tc_fence_after();
            const int64_t row = t.mb * kBM + r_in;
            const bool valid = row < (t.prob == 0 ? p.T : p.Vp);
            const bool pad_row = t.prob == 1 && row >= p.Vr;  // dW rows of padding: exactly 0
            for (int sub = 0; sub < 2 * t.nbox; ++sub) {
                float v[32];
                tmem_ld32(tmem + lane_base + (uint32_t)(acc * kBN + sub * 32), v);
                if (!valid) continue;
                if (pad_row) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = 0.f;
                }
                const int64_t col0 = (int64_t)t.nb * kBN + sub * 32;
                uint16_t* ob = t.prob == 0 ? p.dhidden : p.dw_bf16;
                if (ob) {
                    uint4* o = reinterpret_cast<uint4*>(ob + row * p.H + col0);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        o[q] = make_uint4(pack_bf16x2_rn(v[8 * q], v[8 * q + 1]), pack_bf16x2_rn(v[8 * q + 2], v[8 * q + 3]),
                                          pack_bf16x2_rn(v[8 * q + 4], v[8 * q + 5]),
                                          pack_bf16x2_rn(v[8 * q + 6], v[8 * q + 7]));
                }
                if (t.prob == 1 && p.dw_f32) {
                    float4* o = reinterpret_cast<float4*>(p.dw_f32 + row * p.H + col0);
#pragma unroll
                    for (int q = 0; q < 8; ++q) o[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bars->tempty[acc]));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ----------------------------------------------------------------- host

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
    static std::mutex mu;
    static EncodeTiled fn = nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiled>(ptr);
    }
    return fn;
}

// A BF16 matrix of `rows` rows of `inner` contiguous elements, `stride`
// elements apart, read in boxes of {box_inner, box_rows} with the 128-byte
// swizzle; elements outside [0, inner) x [0, rows) read as zero.
bool make_map(CUtensorMap* m, const void* base, int64_t inner, int64_t rows, int64_t stride, uint32_t box_inner,
              uint32_t box_rows) {
    EncodeTiled enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)stride * 2};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An FP32 matrix [rows, inner] (row-major, inner * 4 bytes a row, a multiple
// of 16) in boxes of box_inner x box_rows with the 128-byte swizzle: the
// stored logits, written by TMA tile stores.
bool make_map_f32(CUtensorMap* m, const void* base, int64_t inner, int64_t rows, uint32_t box_inner,
                  uint32_t box_rows) {
    EncodeTiled enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)inner * 4};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A BF16 matrix whose contiguous dimension `inner` (a multiple of 64) is read
// in 64-element blocks: dims {64, rows, inner/64}, the blocks 128 bytes apart,
// so one box {64, box_rows, box_blocks} lands as box_blocks consecutive
// 64 x box_rows blocks of the 128-byte swizzle -- the layout of as many 2-D
// boxes {64, box_rows}.  Blocks past inner/64 read as zero.
bool make_map_mn3(CUtensorMap* m, const void* base, int64_t inner, int64_t rows, int64_t stride, uint32_t box_rows,
                  uint32_t box_blocks) {
    EncodeTiled enc = encode_fn();
    if (!enc || inner % 64 != 0) return false;
    const cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)(inner / 64)};
    const cuuint64_t strides[2] = {(cuuint64_t)stride * 2, 128};
    const cuuint32_t box[3] = {64, box_rows, box_blocks};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

constexpr size_t kGemmSmem = 1024 + kGemmSmemCore;
// kEpiPartialsStore adds one 32 x 33 FP32 staging block per epilogue warp.
constexpr size_t kGemmSmemStore = kGemmSmem + 4 * kStoreStage * sizeof(float);
static_assert(kStoreStage * sizeof(float) % 1024 == 0 && kStoreStage >= 32 * 33, "staging block per warp");

// Chunks of kBN weight rows per tile (the last one may be narrower).
int64_t chunks_per_tile(const rlk_logp_contract& c) { return (c.V_padded / c.num_tiles + kBN - 1) / kBN; }

size_t partial_bytes(const rlk_logp_contract& c) {
    return round256((size_t)c.T * c.num_tiles * chunks_per_tile(c) * 8);
}

size_t dlogits_bytes(const rlk_logp_contract& c) { return round256((size_t)c.T * c.V_padded * 2); }

}  // namespace

// Workspace beyond the status word: tickets, FP32 chunk partials
// [T, NT * chunks, 2], target logits [T]; the backward adds BF16 dlogits
// [T, V_padded] and, for the forward+backward in one call, the forward's FP32
// logits [T, V_padded].
size_t lmhead_fwd_workspace(const rlk_logp_contract& c) {
    return kTicketBytes + partial_bytes(c) + round256((size_t)c.T * 4);
}

size_t lmhead_bwd_workspace(const rlk_logp_contract& c) {
    return lmhead_fwd_workspace(c) + dlogits_bytes(c) + round256((size_t)c.T * c.V_padded * 4);
}

rlk_status lmhead_check(const rlk_logp_contract& c, int64_t H) {
    if (H < kBK || H % kBK != 0) return fail(RLK_ERR_UNSUPPORTED, "hidden size H must be a positive multiple of 64");
    if (H > (int64_t)1 << 20) return fail(RLK_ERR_UNSUPPORTED, "hidden size H above 2^20");
    const int64_t W = c.V_padded / c.num_tiles;
    if (W % 16 != 0) return fail(RLK_ERR_UNSUPPORTED, "the fused lm_head needs a tile width that is a multiple of 16");
    if (c.T > ((int64_t)1 << 31) - kBM) return fail(RLK_ERR_UNSUPPORTED, "T above 2^31 rows for the fused lm_head");
    return RLK_OK;
}

namespace {

struct LmLaunch {
    LmParams p;
    CUtensorMap tmH, tmW, tmWr;
    int grid, sms;
};

rlk_status sm_count(int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || *sms <= 0)
        return fail(RLK_ERR_CUDA, "cannot query the device's SM count");
    return RLK_OK;
}

rlk_status prepare(LmLaunch& L, const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                   const int64_t* targets, const uint8_t* mask, uint32_t* status, unsigned long long* tickets) {
    int sms = 0;
    rlk_status st = sm_count(&sms);
    if (st != RLK_OK) return st;
    LmParams& p = L.p;
    p = LmParams{};
    p.targets = targets;
    p.mask = mask;
    p.tickets = tickets;
    p.w.status = status;
    p.w.wait_ns = c.wait_timeout_ns > 0 ? (uint64_t)c.wait_timeout_ns : kDefaultWaitNs;
    p.T = c.T;
    p.Vr = c.V_real;
    p.Vp = c.V_padded;
    p.ignore_index = c.ignore_index;
    p.K = (int32_t)H;
    p.NT = c.num_tiles;
    p.W = (int32_t)(c.V_padded / c.num_tiles);
    p.vtp = c.virtual_tp;
    p.nchunk = (p.W + kBN - 1) / kBN;
    p.rem = p.W % kBN;
    p.mask_mode = c.mask_mode;
    p.MB = (int32_t)((c.T + kBM - 1) / kBM);
    {
        const int64_t band = kBandHiddenBytes / ((int64_t)kBM * H * 2);
        p.MBg = (int32_t)(band < 1 ? 1 : band < p.MB ? band : p.MB);
    }
    p.keep_hidden = kKeepHidden;
    const uint32_t rrows = p.rem ? (uint32_t)p.rem : (uint32_t)kBN;
    if (!make_map(&L.tmH, hidden, H, c.T, H, kBK, kBM) || !make_map(&L.tmW, weight, H, c.V_padded, H, kBK, kBN) ||
        !make_map(&L.tmWr, weight, H, c.V_padded, H, kBK, rrows))
        return fail(RLK_ERR_CUDA, "cuTensorMapEncodeTiled failed for the hidden or weight tensor");
    const int64_t units_per_shard = (int64_t)(c.num_tiles / c.virtual_tp) * p.nchunk * p.MB;
    int64_t per_group = sms / c.virtual_tp;  // CTAs per virtual-TP group
    if (per_group > units_per_shard) per_group = units_per_shard;
    if (per_group < 1) per_group = 1;
    L.grid = (int)(per_group * c.virtual_tp);
    L.sms = sms;
    return RLK_OK;
}

template <class K, class... Args>
rlk_status launch_gemm_smem(K kernel, int grid, size_t smem, cudaStream_t stream, const char* what, Args... args) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
    kernel<<<(unsigned)grid, kThreadsLm, smem, stream>>>(args...);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string(what) + " launch: " + cudaGetErrorString(e));
    return RLK_OK;
}

template <class K, class... Args>
rlk_status launch_gemm(K kernel, int grid, cudaStream_t stream, const char* what, Args... args) {
    return launch_gemm_smem(kernel, grid, kGemmSmem, stream, what, args...);
}

rlk_status clear_tickets(void* tickets, cudaStream_t stream) {
    const cudaError_t e = cudaMemsetAsync(tickets, 0, kTicketBytes, stream);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("clearing the tickets: ") + cudaGetErrorString(e));
    return RLK_OK;
}

// The forward: the logits GEMM with the partials epilogue (and, with xlog,
// the FP32 logits stored), then the fold.
rlk_status forward(const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                   const int64_t* targets, const uint8_t* mask, float* logp, float* lse, void* workspace,
                   float* xlog, uint32_t* status, cudaStream_t stream) {
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    unsigned long long* tickets = reinterpret_cast<unsigned long long*>(ws);
    rlk_status st = clear_tickets(tickets, stream);
    if (st != RLK_OK) return st;
    LmLaunch L;
    if ((st = prepare(L, c, hidden, H, weight, targets, mask, status, tickets)) != RLK_OK) return st;
    LmParams& p = L.p;
    p.partials = reinterpret_cast<float2*>(ws + kTicketBytes);
    p.xt = reinterpret_cast<float*>(ws + kTicketBytes + partial_bytes(c));
    p.xlog = xlog;
    if (xlog) {
        // the FP32 logits [T, V_padded]: 32 x 32 boxes with the 128-byte swizzle
        CUtensorMap tmX;
        if (!make_map_f32(&tmX, xlog, c.V_padded, c.T, 32, 32))
            return fail(RLK_ERR_CUDA, "cuTensorMapEncodeTiled failed for the stored logits");
        st = launch_gemm_smem(lmhead_kernel<kEpiPartialsStore>, L.grid, kGemmSmemStore, stream, "lm_head GEMM", L.tmH,
                              L.tmW, L.tmWr, tmX, p);
    } else {
        st = launch_gemm(lmhead_kernel<kEpiPartials>, L.grid, stream, "lm_head GEMM", L.tmH, L.tmW, L.tmWr, L.tmH, p);
    }
    if (st != RLK_OK) return st;
    const int fold_threads = 256;
    const size_t fold_smem = (size_t)(fold_threads / 32) * c.num_tiles * sizeof(float2);
    cudaError_t e =
        cudaFuncSetAttribute(lmhead_fold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fold_smem);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
    int64_t fold_grid = (c.T + 7) / 8;
    if (fold_grid > (int64_t)L.sms * 8) fold_grid = (int64_t)L.sms * 8;
    lmhead_fold_kernel<<<(unsigned)fold_grid, fold_threads, fold_smem, stream>>>(
        p.partials, p.xt, targets, mask, c.mask_mode, c.ignore_index, c.T, c.V_real, c.num_tiles, p.nchunk, logp, lse,
        status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("lm_head fold launch: ") + cudaGetErrorString(e));
    return RLK_OK;
}

// dHidden = dlogits[:, :V_real] W[:V_real] and dW = dlogits[:, :V_real]^T hidden in one launch.
// The maps stop at V_real (and at T), so padded columns of dlogits, padded
// rows of W and rows past T read as zero; rows [V_real, V_padded) of dW come
// out exactly 0.
rlk_status grad_gemms(const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                      const uint16_t* dlogits, void* dhidden, float* dweight_f32, void* dweight_bf16,
                      unsigned long long* ticket, uint32_t* status, cudaStream_t stream) {
    int sms = 0;
    rlk_status st = sm_count(&sms);
    if (st != RLK_OK) return st;
    CUtensorMap tmA0, tmB0, tmA1, tmB1;
    if (!make_map(&tmA0, dlogits, c.V_real, c.T, c.V_padded, kBK, kBM) ||
        !make_map_mn3(&tmB0, weight, H, c.V_real, H, kBK, 4) ||
        !make_map(&tmA1, dlogits, c.V_real, c.T, c.V_padded, 64, kBK) ||
        !make_map_mn3(&tmB1, hidden, H, c.T, H, kBK, 4))
        return fail(RLK_ERR_CUDA, "cuTensorMapEncodeTiled failed for a gradient operand");
    GradParams g{};
    g.dhidden = static_cast<uint16_t*>(dhidden);
    g.dw_bf16 = static_cast<uint16_t*>(dweight_bf16);
    g.dw_f32 = dweight_f32;
    g.ticket = ticket;
    g.w.status = status;
    g.w.wait_ns = c.wait_timeout_ns > 0 ? (uint64_t)c.wait_timeout_ns : kDefaultWaitNs;
    g.T = c.T;
    g.Vr = c.V_real;
    g.Vp = c.V_padded;
    g.H = (int32_t)H;
    g.NB = (int32_t)((H + kBN - 1) / kBN);
    g.KB0 = (int32_t)((c.V_real + kBK - 1) / kBK);
    g.KB1 = (int32_t)((c.T + kBK - 1) / kBK);
    g.NBg = g.NB < kBandN ? g.NB : kBandN;
    g.n0 = ((c.T + kBM - 1) / kBM) * g.NB;
    g.n1 = ((c.V_padded + kBM - 1) / kBM) * g.NB;
    const int64_t total = g.n0 + g.n1;
    const int grid = (int)(total < sms ? total : sms);
    return launch_gemm(lmhead_grad_kernel, grid, stream, "lm_head gradient GEMM", tmA0, tmB0, tmA1, tmB1, g);
}

// dlogits = g * (onehot - exp(x - LSE)) from FP32 logits (BF16 [T, V_padded]
// in the workspace), then dHidden and dW.  The gradient GEMM's ticket must be
// zero at entry.
rlk_status backward_from_logits(const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                                const int64_t* targets, const uint8_t* mask, const float* grad, const float* lse,
                                const float* xlog, void* dhidden, float* dweight_f32, void* dweight_bf16,
                                void* workspace, uint32_t* status, cudaStream_t stream) {
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    uint16_t* dlogits = reinterpret_cast<uint16_t*>(ws + lmhead_fwd_workspace(c));
    // one block a row (the hardware balances the tail), at most 2^31 - 1 blocks
    const int64_t grid = c.T < 0x7FFFFFFF ? c.T : 0x7FFFFFFF;
    lmhead_dlogits_kernel<<<(unsigned)grid, 256, 0, stream>>>(xlog, lse, grad, targets, mask, c.mask_mode,
                                                              c.ignore_index, c.T, c.V_real, c.V_padded, dlogits,
                                                              status);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("lm_head dlogits launch: ") + cudaGetErrorString(e));
    unsigned long long* tickets = reinterpret_cast<unsigned long long*>(ws);
    return grad_gemms(c, hidden, H, weight, dlogits, dhidden, dweight_f32, dweight_bf16, tickets + 2 * kMaxGroups,
                      status, stream);
}

}  // namespace

rlk_status launch_lmhead_fwd(const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                             const int64_t* targets, const uint8_t* mask, float* logp, float* lse, void* workspace,
                             uint32_t* status, cudaStream_t stream) {
    return forward(c, hidden, H, weight, targets, mask, logp, lse, workspace, nullptr, status, stream);
}

// Forward and backward in one call: the forward stores its FP32 logits in the
// workspace (the accumulators the recompute GEMM would form again, bitwise),
// an elementwise pass turns them into dlogits with the forward's LSE, then the
// gradient GEMMs.
rlk_status launch_lmhead_bwd(const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                             const int64_t* targets, const uint8_t* mask, const float* grad, float* logp, float* lse,
                             void* dhidden, float* dweight_f32, void* dweight_bf16, void* workspace, uint32_t* status,
                             cudaStream_t stream) {
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    float* xlog = reinterpret_cast<float*>(ws + lmhead_fwd_workspace(c) + dlogits_bytes(c));
    // the forward clears every ticket, the gradient GEMM's among them
    rlk_status st = forward(c, hidden, H, weight, targets, mask, logp, lse, workspace, xlog, status, stream);
    if (st != RLK_OK) return st;
    return backward_from_logits(c, hidden, H, weight, targets, mask, grad, lse, xlog, dhidden, dweight_f32,
                                dweight_bf16, workspace, status, stream);
}

rlk_status launch_lmhead_fwd_keep(const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                                  const int64_t* targets, const uint8_t* mask, float* logp, float* lse,
                                  float* logits_f32, void* workspace, uint32_t* status, cudaStream_t stream) {
    return forward(c, hidden, H, weight, targets, mask, logp, lse, workspace, logits_f32, status, stream);
}

rlk_status launch_lmhead_bwd_kept(const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                                  const int64_t* targets, const uint8_t* mask, const float* grad, const float* lse,
                                  const float* logits_f32, void* dhidden, float* dweight_f32, void* dweight_bf16,
                                  void* workspace, uint32_t* status, cudaStream_t stream) {
    rlk_status st = clear_tickets(workspace, stream);
    if (st != RLK_OK) return st;
    return backward_from_logits(c, hidden, H, weight, targets, mask, grad, lse, logits_f32, dhidden, dweight_f32,
                                dweight_bf16, workspace, status, stream);
}

// The backward alone, from a given LSE: the recompute GEMM's epilogue forms
// dlogits, then the gradient GEMMs.
rlk_status launch_lmhead_bwd_given_lse(const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                                       const int64_t* targets, const uint8_t* mask, const float* grad,
                                       const float* lse, void* dhidden, float* dweight_f32, void* dweight_bf16,
                                       void* workspace, uint32_t* status, cudaStream_t stream) {
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    unsigned long long* tickets = reinterpret_cast<unsigned long long*>(ws);
    rlk_status st = clear_tickets(tickets, stream);
    if (st != RLK_OK) return st;
    uint16_t* dlogits = reinterpret_cast<uint16_t*>(ws + lmhead_fwd_workspace(c));
    // dlogits = g * (onehot - exp(x - LSE)) from the recomputed logits (BF16 [T, V_padded])
    LmLaunch L;
    if ((st = prepare(L, c, hidden, H, weight, targets, mask, status, tickets + kMaxGroups)) != RLK_OK) return st;
    L.p.lse_in = lse;
    L.p.grad = grad;
    L.p.dlogits = dlogits;
    if ((st = launch_gemm(lmhead_kernel<kEpiGrad>, L.grid, stream, "lm_head recompute GEMM", L.tmH, L.tmW, L.tmWr,
                          L.tmH, L.p)) != RLK_OK)
        return st;
    return grad_gemms(c, hidden, H, weight, dlogits, dhidden, dweight_f32, dweight_bf16, tickets + 2 * kMaxGroups,
                      status, stream);
}

}  // namespace rlk
