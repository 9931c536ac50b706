// Fused lm_head variant (sm_103a): the selected-token log-probability of
// logits = hidden @ W^T without materialising the logits.
//
// The optional fused kernel of issue #323 ("[WS2][Logprob] H100 validation
// and reproduction guide", "Validation Boundary": "the optional PR6 fused
// kernel") is the prior art; its design is not on the pages.  Here each
// (128-token block, global vocabulary tile) unit runs a tcgen05 GEMM over the
// tile's columns in chunks of up to 256 vocabulary rows (accumulators in
// tensor memory, operands staged by TMA with the 128-byte swizzle), and the
// epilogue turns each chunk into the running (max, sumexp) partial of the
// tile -- the same per-tile partials as the streaming path, but of FP32
// logits that are never rounded or written.  A fold kernel then merges the
// tiles in fixed index order (rlk_fold.cuh) and forms logp.
//
// Roles (192 threads, one CTA per SM): warp 0 issues the TMA loads, warp 1
// allocates tensor memory and issues the MMAs, warps 2-5 run the epilogue
// (warp w reads TMEM lanes 32*(w%4)..+31, one token row per thread).
// Virtual TP: the CTAs are split into virtual_tp groups; group j computes
// only the tiles of vocabulary shard j.  A tile's partial is computed by one
// thread in one fixed order (chunks, then 32-column blocks, then columns),
// whatever the grouping, so outputs do not depend on virtual_tp.
//
// Every wait is bounded; on expiry the CTA records RLK_ERR_TIMEOUT, stops
// issuing, waits (bounded) for its issued copies and MMAs, frees its tensor
// memory and returns.
#include <cublasLt.h>
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <cstdlib>
#include <mutex>
#include <string>

#include "rlk_fold.cuh"
#include "rlk_internal.h"
#include "rlk_ptx.cuh"

namespace rlk {
namespace {

int env_int_lm(const char* name, int dflt) {
    const char* v = std::getenv(name);
    return (v && *v) ? std::atoi(v) : dflt;
}

constexpr int kBM = 128;  // token rows per unit (TMEM lanes)
constexpr int kBN = 256;  // vocabulary rows per chunk (accumulator columns)
constexpr int kBK = 64;   // K per stage: 64 BF16 = one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kThreadsLm = 192;
constexpr uint32_t kTmemCols = 512;  // two accumulators of kBN columns
constexpr uint32_t kStageA = kBM * kBK * 2;
constexpr uint32_t kStageB = kBN * kBK * 2;
constexpr uint64_t kDrainNsLm = 1000000000ull;

enum : int { kEpiPartials = 0, kEpiGrad = 1 };

struct LmParams {
    const int64_t* targets;
    const uint8_t* mask;
    float2* partials;  // [T, NT]                     (kEpiPartials)
    float* xt;         // [T] target logits          (kEpiPartials)
    const float* lse_in;  // [T]                      (kEpiGrad)
    const float* grad;    // [T] upstream g of logp   (kEpiGrad)
    uint16_t* dlogits;    // [T, Vp] BF16 out         (kEpiGrad)
    uint32_t* status;
    int64_t T, Vr, Vp, ignore_index;
    uint64_t wait_ns;
    int32_t K, NT, W, vtp, nchunk, rem, mask_mode;
    int32_t MB;    // token blocks
    int32_t pair;  // CTAs per cluster: 2 = two token blocks share each weight chunk (multicast), else 1
};

struct Bars {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t drain;
    uint32_t tmem_addr;
    int abort_flag;
};

// Units of this CTA: the tiles of its virtual-TP shard times the token
// blocks, tile-major, strided over the clusters of its group.  With pairs
// (p.pair = 2) a unit is a tile times a pair of token blocks: rank r of the
// cluster takes block 2i + r (which may lie past the last block; its rows
// are then out of range and masked).  The group of a cluster is a
// contiguous run of clusters, so both ranks see the same units.
struct UnitSeq {
    int64_t u, step, end;
    int tile0, ntile_sh, MBU, rank, pair;
    __device__ void init(const LmParams& p) {
        pair = p.pair;
        const int cl = blockIdx.x / pair;
        rank = blockIdx.x % pair;
        const int G = gridDim.x / pair;
        const int Gj = G / p.vtp;
        const int j = cl / Gj;
        const int c = cl % Gj;
        ntile_sh = p.NT / p.vtp;
        tile0 = j * ntile_sh;
        MBU = (p.MB + pair - 1) / pair;
        u = c;
        step = Gj;
        end = (int64_t)ntile_sh * MBU;
    }
    __device__ bool next(int& tile, int& mb) {
        if (u >= end) return false;
        tile = tile0 + (int)(u / MBU);
        mb = (int)(u % MBU) * pair + rank;
        u += step;
        return true;
    }
};

__device__ bool lm_wait(Bars* bars, uint32_t bar, uint32_t parity, const LmParams& p) {
    if (mbar_try_wait(bar, parity)) return true;
    volatile int* ab = &bars->abort_flag;
    if (*ab) return false;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*ab) return false;
        if (globaltimer_ns() - t0 > p.wait_ns) {
            *ab = 1;
            atomicOr(p.status, kStatusTimeout);
            return false;
        }
    }
}

__device__ void lm_drain_wait(uint32_t bar, uint32_t parity, const LmParams& p) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kDrainNsLm) {
            atomicOr(p.status, kStatusTimeout);
            return;
        }
    }
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
                      const __grid_constant__ CUtensorMap tmWr, const __grid_constant__ LmParams p) {
    // With pairs, tmW and tmWr describe half a chunk (128 rows, rem/2 rows):
    // each rank loads its half and multicasts it to both CTAs.
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte alignment for the 128-byte-swizzled operand tiles.
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* sA = smem;
    unsigned char* sB = smem + kStages * kStageA;
    Bars* bars = reinterpret_cast<Bars*>(smem + kStages * (kStageA + kStageB));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int KB = p.K / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&bars->full[s]), 1);
            // with pairs a stage is free once both CTAs' MMAs have read it
            mbar_init(smem_u32(&bars->empty[s]), (uint32_t)p.pair);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bars->tfull[b]), 1);
            mbar_init(smem_u32(&bars->tempty[b]), 4);
        }
        mbar_init(smem_u32(&bars->drain), 1);
        bars->abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&bars->tmem_addr), kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    // the peer's barriers must be initialised before any multicast or commit reaches them
    if (p.pair > 1) cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem = bars->tmem_addr;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            UnitSeq us;
            us.init(p);
            int tile, mb, stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool aborted = false;
            while (!aborted && us.next(tile, mb)) {
                for (int ch = 0; ch < p.nchunk && !aborted; ++ch) {
                    const bool last_rem = (ch == p.nchunk - 1) && p.rem;
                    const int nrows = last_rem ? p.rem : kBN;
                    const int n0 = tile * p.W + ch * kBN;
                    for (int kb = 0; kb < KB; ++kb) {
                        const uint32_t eb = smem_u32(&bars->empty[stage]);
                        if (!lm_wait(bars, eb, phase ^ 1u, p)) {
                            aborted = true;
                            break;
                        }
                        const uint32_t fb = smem_u32(&bars->full[stage]);
                        mbar_arrive_expect_tx(fb, kStageA + (uint32_t)nrows * kBK * 2);
                        tma_load_2d(smem_u32(sA + stage * kStageA), &tmH, kb * kBK, mb * kBM, fb);
                        if (p.pair == 1) {
                            tma_load_2d(smem_u32(sB + stage * kStageB), last_rem ? &tmWr : &tmW, kb * kBK, n0, fb);
                        } else {
                            // rows [rank*half, (rank+1)*half) of the chunk, to both CTAs
                            const int half = nrows / 2;
                            tma_load_2d_mc(smem_u32(sB + stage * kStageB + us.rank * half * (kBK * 2)),
                                           last_rem ? &tmWr : &tmW, kb * kBK, n0 + us.rank * half, fb, 0x3);
                        }
                        ++issued;
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                }
            }
            // Drain: every issued copy lands before this CTA may exit.
            const int64_t first = issued > kStages ? issued - kStages : 0;
            for (int64_t j = first; j < issued; ++j)
                lm_drain_wait(smem_u32(&bars->full[j % kStages]), (uint32_t)((j / kStages) & 1), p);
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            UnitSeq us;
            us.init(p);
            int tile, mb, stage = 0;
            uint32_t phase = 0;
            int64_t chunk = 0;
            bool aborted = false;
            while (!aborted && us.next(tile, mb)) {
                for (int ch = 0; ch < p.nchunk && !aborted; ++ch, ++chunk) {
                    const int acc = (int)(chunk & 1);
                    const uint32_t accph = (uint32_t)((chunk >> 1) & 1);
                    if (!lm_wait(bars, smem_u32(&bars->tempty[acc]), accph ^ 1u, p)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
                    const bool last_rem = (ch == p.nchunk - 1) && p.rem;
                    const uint32_t idesc = idesc_bf16_f32(kBM, last_rem ? (uint32_t)p.rem : (uint32_t)kBN);
                    const uint32_t d = tmem + (uint32_t)(acc * kBN);
                    for (int kb = 0; kb < KB; ++kb) {
                        if (!lm_wait(bars, smem_u32(&bars->full[stage]), phase, p)) {
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
                        // frees the stage (in both CTAs of a pair) when these MMAs finish
                        if (p.pair == 1)
                            umma_commit(smem_u32(&bars->empty[stage]));
                        else
                            umma_commit_mc(smem_u32(&bars->empty[stage]), 0x3);
                        if (++stage == kStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                    if (!aborted) umma_commit(smem_u32(&bars->tfull[acc]));
                }
            }
            // Every issued MMA completes before tensor memory is freed.
            umma_commit(smem_u32(&bars->drain));
            lm_drain_wait(smem_u32(&bars->drain), 0u, p);
        }
    } else {
        // ------------------------------------------------ epilogue (warps 2..5)
        const int quarter = warp & 3;
        const int r_in = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        UnitSeq us;
        us.init(p);
        int tile, mb;
        int64_t chunk = 0;
        bool aborted = false;
        while (!aborted && us.next(tile, mb)) {
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
                nlL = -__fmul_rn(p.lse_in[row], kLog2e);
                drow = p.dlogits + row * p.Vp;
            }
            for (int ch = 0; ch < p.nchunk; ++ch, ++chunk) {
                const int acc = (int)(chunk & 1);
                const uint32_t accph = (uint32_t)((chunk >> 1) & 1);
                const bool ok = lm_wait(bars, smem_u32(&bars->tfull[acc]), accph, p);
                if (!__all_sync(0xFFFFFFFFu, ok)) {
                    aborted = true;
                    break;
                }
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
            }
            if (EPI == kEpiPartials && !aborted && valid) {
                p.partials[row * p.NT + tile] = make_float2(m_run, s_run);
                if (have_xt) p.xt[row] = xt;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    // no CTA of a pair leaves while the other may still multicast or commit into it
    if (p.pair > 1) cluster_sync_all();
}

// LSE and logp of each row from its tile partials (one warp per row).
__global__ void lmhead_fold_kernel(const float2* partials, const float* xt, const int64_t* targets,
                                   const uint8_t* mask, int mask_mode, int64_t ignore_index, int64_t T, int64_t Vr,
                                   int NT, float* logp, float* lse, uint32_t* status) {
    extern __shared__ float2 scratch[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int wpb = blockDim.x >> 5;
    float2* sc = scratch + (size_t)warp * NT;
    for (int64_t row = (int64_t)blockIdx.x * wpb + warp; row < T; row += (int64_t)gridDim.x * wpb) {
        const float l = fold_tiles(partials + row * NT, NT, sc, lane);
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

// K-major [rows, K] BF16 matrix, box {64, box_rows}, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t K, uint32_t box_rows) {
    EncodeTiled enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t lmhead_fwd_workspace(const rlk_logp_contract& c) {
    return ((size_t)c.T * c.num_tiles * 8 + 255) / 256 * 256 + ((size_t)c.T * 4 + 255) / 256 * 256;
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

// Pairs of CTAs share each weight chunk when every virtual-TP group gets a
// whole number of pairs on the SMs (all but virtual TP 8 on 152 SMs); the
// number of pairs per group stays within the group's units.

rlk_status prepare(LmLaunch& L, const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                   const int64_t* targets, const uint8_t* mask, uint32_t* status) {
    int dev = 0;
    cudaGetDevice(&dev);
    int sms = 0;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    LmParams& p = L.p;
    p = LmParams{};
    p.targets = targets;
    p.mask = mask;
    p.status = status;
    p.T = c.T;
    p.Vr = c.V_real;
    p.Vp = c.V_padded;
    p.ignore_index = c.ignore_index;
    p.wait_ns = c.wait_timeout_ns > 0 ? (uint64_t)c.wait_timeout_ns : kDefaultWaitNs;
    p.K = (int32_t)H;
    p.NT = c.num_tiles;
    p.W = (int32_t)(c.V_padded / c.num_tiles);
    p.vtp = c.virtual_tp;
    p.nchunk = (p.W + kBN - 1) / kBN;
    p.rem = p.W % kBN;
    p.mask_mode = c.mask_mode;
    p.MB = (int32_t)((c.T + kBM - 1) / kBM);
    const int forced = env_int_lm("RLK_LMHEAD_PAIR", 0);
    p.pair = ((sms / 2) % c.virtual_tp == 0 && p.MB >= 2) ? 2 : 1;
    if (forced == 1 || forced == 2) p.pair = forced;
    const uint32_t brows = p.pair == 2 ? kBN / 2 : kBN;
    const uint32_t rrows = p.rem ? (uint32_t)p.rem / (uint32_t)p.pair : brows;
    if (!make_map(&L.tmH, hidden, c.T, H, kBM) || !make_map(&L.tmW, weight, c.V_padded, H, brows) ||
        !make_map(&L.tmWr, weight, c.V_padded, H, rrows))
        return fail(RLK_ERR_CUDA, "cuTensorMapEncodeTiled failed for the hidden or weight tensor");
    const int64_t units_per_shard = (int64_t)(c.num_tiles / c.virtual_tp) * ((p.MB + p.pair - 1) / p.pair);
    int64_t per_group = sms / p.pair / c.virtual_tp;  // clusters per virtual-TP group
    if (per_group > units_per_shard) per_group = units_per_shard;
    if (per_group < 1) per_group = 1;
    L.grid = (int)(per_group * c.virtual_tp * p.pair);
    L.sms = sms;
    return RLK_OK;
}

template <int EPI>
rlk_status run_gemm(const LmLaunch& L, cudaStream_t stream) {
    const size_t smem = 1024 + (size_t)kStages * (kStageA + kStageB) + sizeof(Bars);
    cudaError_t e = cudaFuncSetAttribute(lmhead_kernel<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
    cudaLaunchConfig_t cfg{};
    cudaLaunchAttribute attr[1];
    cfg.gridDim = dim3((unsigned)L.grid, 1, 1);
    cfg.blockDim = dim3(kThreadsLm, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.numAttrs = 0;
    if (L.p.pair > 1) {
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)L.p.pair;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        // The two CTAs of a pair wait on each other; the hardware schedules a
        // cluster's CTAs together, and pairs never wait on other pairs.
    }
    e = cudaLaunchKernelEx(&cfg, lmhead_kernel<EPI>, L.tmH, L.tmW, L.tmWr, L.p);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("lm_head GEMM launch: ") + cudaGetErrorString(e));
    return RLK_OK;
}

}  // namespace

rlk_status launch_lmhead_fwd(const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                             const int64_t* targets, const uint8_t* mask, float* logp, float* lse, void* workspace,
                             uint32_t* status, cudaStream_t stream) {
    LmLaunch L;
    rlk_status st = prepare(L, c, hidden, H, weight, targets, mask, status);
    if (st != RLK_OK) return st;
    LmParams& p = L.p;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    p.partials = reinterpret_cast<float2*>(ws);
    p.xt = reinterpret_cast<float*>(ws + ((size_t)c.T * c.num_tiles * 8 + 255) / 256 * 256);
    if ((st = run_gemm<kEpiPartials>(L, stream)) != RLK_OK) return st;
    const int sms = L.sms;
    cudaError_t e;
    int dev = 0;
    cudaGetDevice(&dev);
    (void)dev;
    const int fold_threads = 256;
    const size_t fold_smem = (size_t)(fold_threads / 32) * c.num_tiles * sizeof(float2);
    e = cudaFuncSetAttribute(lmhead_fold_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fold_smem);
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("cudaFuncSetAttribute: ") + cudaGetErrorString(e));
    int64_t fold_grid = (c.T + 7) / 8;
    if (fold_grid > (int64_t)sms * 8) fold_grid = (int64_t)sms * 8;
    lmhead_fold_kernel<<<(unsigned)fold_grid, fold_threads, fold_smem, stream>>>(
        p.partials, p.xt, targets, mask, c.mask_mode, c.ignore_index, c.T, c.V_real, c.num_tiles, logp, lse, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("lm_head fold launch: ") + cudaGetErrorString(e));
    return RLK_OK;
}

// ----------------------------------------------------------------- backward

namespace {

constexpr size_t kLtWorkspace = (size_t)32 << 20;

cublasLtHandle_t lt_handle(int dev) {
    static std::mutex mu;
    static cublasLtHandle_t handles[64] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return nullptr;
    if (!handles[dev] && cublasLtCreate(&handles[dev]) != CUBLAS_STATUS_SUCCESS) handles[dev] = nullptr;
    return handles[dev];
}

// C[m, n] = op(A) op(B) in column-major terms, BF16 in and out, FP32 accumulate;
// reductions across K chunks are excluded, so every output element is summed in
// one fixed order (deterministic, no atomics).
rlk_status lt_gemm(cublasLtHandle_t h, cublasOperation_t opA, cublasOperation_t opB, uint64_t m, uint64_t n,
                   uint64_t k, const void* A, int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                   void* ws, cudaStream_t stream) {
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
    cublasLtMatmulPreference_t pref = nullptr;
    rlk_status st = RLK_OK;
    auto ok = [&](cublasStatus_t s, const char* what) {
        if (s != CUBLAS_STATUS_SUCCESS && st == RLK_OK) st = fail(RLK_ERR_CUDA, std::string("cuBLASLt ") + what);
        return st == RLK_OK;
    };
    const uint32_t scheme = CUBLASLT_REDUCTION_SCHEME_NONE;
    const uint64_t wsb = kLtWorkspace;
    if (ok(cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F), "desc") &&
        ok(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSA, &opA, sizeof(opA)), "transa") &&
        ok(cublasLtMatmulDescSetAttribute(op, CUBLASLT_MATMUL_DESC_TRANSB, &opB, sizeof(opB)), "transb") &&
        ok(cublasLtMatrixLayoutCreate(&la, CUDA_R_16BF, opA == CUBLAS_OP_N ? m : k, opA == CUBLAS_OP_N ? k : m, lda),
           "layout A") &&
        ok(cublasLtMatrixLayoutCreate(&lb, CUDA_R_16BF, opB == CUBLAS_OP_N ? k : n, opB == CUBLAS_OP_N ? n : k, ldb),
           "layout B") &&
        ok(cublasLtMatrixLayoutCreate(&lc, CUDA_R_16BF, m, n, ldc), "layout C") &&
        ok(cublasLtMatmulPreferenceCreate(&pref), "preference") &&
        ok(cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &wsb, sizeof(wsb)),
           "workspace pref") &&
        ok(cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_REDUCTION_SCHEME_MASK, &scheme,
                                                sizeof(scheme)),
           "reduction pref")) {
        cublasLtMatmulHeuristicResult_t res{};
        int found = 0;
        if (ok(cublasLtMatmulAlgoGetHeuristic(h, op, la, lb, lc, lc, pref, 1, &res, &found), "heuristic")) {
            if (found < 1) {
                st = fail(RLK_ERR_UNSUPPORTED, "cuBLASLt found no deterministic algorithm for the lm_head backward");
            } else {
                const float alpha = 1.f, beta = 0.f;
                ok(cublasLtMatmul(h, op, &alpha, A, la, B, lb, &beta, C, lc, C, lc, &res.algo, ws, kLtWorkspace, stream),
                   "matmul");
            }
        }
    }
    if (pref) cublasLtMatmulPreferenceDestroy(pref);
    if (lc) cublasLtMatrixLayoutDestroy(lc);
    if (lb) cublasLtMatrixLayoutDestroy(lb);
    if (la) cublasLtMatrixLayoutDestroy(la);
    if (op) cublasLtMatmulDescDestroy(op);
    return st;
}

}  // namespace

size_t lmhead_bwd_workspace(const rlk_logp_contract& c) {
    return lmhead_fwd_workspace(c) + ((size_t)c.T * c.V_padded * 2 + 255) / 256 * 256 + kLtWorkspace;
}

rlk_status launch_lmhead_bwd(const rlk_logp_contract& c, const void* hidden, int64_t H, const void* weight,
                             const int64_t* targets, const uint8_t* mask, const float* grad, float* logp, float* lse,
                             void* dhidden, void* dweight, void* workspace, uint32_t* status, cudaStream_t stream) {
    rlk_status st = launch_lmhead_fwd(c, hidden, H, weight, targets, mask, logp, lse, workspace, status, stream);
    if (st != RLK_OK) return st;
    unsigned char* ws = static_cast<unsigned char*>(workspace) + lmhead_fwd_workspace(c);
    uint16_t* dlogits = reinterpret_cast<uint16_t*>(ws);
    void* lt_ws = ws + ((size_t)c.T * c.V_padded * 2 + 255) / 256 * 256;
    // dlogits = g * (onehot - exp(x - LSE)) from the recomputed logits (BF16 [T, V_padded]).
    LmLaunch L;
    if ((st = prepare(L, c, hidden, H, weight, targets, mask, status)) != RLK_OK) return st;
    L.p.lse_in = lse;
    L.p.grad = grad;
    L.p.dlogits = dlogits;
    if ((st = run_gemm<kEpiGrad>(L, stream)) != RLK_OK) return st;
    int dev = 0;
    cudaGetDevice(&dev);
    cublasLtHandle_t h = lt_handle(dev);
    if (!h) return fail(RLK_ERR_CUDA, "cublasLtCreate failed");
    // dHidden [T, H] = dlogits[:, :V_real] W[:V_real]; column-major: [H, T] = W_cm[H, Vr] x dlogits_cm[Vr, T].
    if ((st = lt_gemm(h, CUBLAS_OP_N, CUBLAS_OP_N, (uint64_t)H, (uint64_t)c.T, (uint64_t)c.V_real, weight, H, dlogits,
                      c.V_padded, dhidden, H, lt_ws, stream)) != RLK_OK)
        return st;
    // dW[:V_real] = dlogits[:, :V_real]^T hidden; column-major: [H, Vr] = hidden_cm[H, T] x (dlogits_cm[Vr, T])^T.
    if ((st = lt_gemm(h, CUBLAS_OP_N, CUBLAS_OP_T, (uint64_t)H, (uint64_t)c.V_real, (uint64_t)c.T, hidden, H, dlogits,
                      c.V_padded, dweight, H, lt_ws, stream)) != RLK_OK)
        return st;
    if (c.V_padded > c.V_real) {
        const cudaError_t e = cudaMemsetAsync(static_cast<uint16_t*>(dweight) + (size_t)c.V_real * H, 0,
                                              (size_t)(c.V_padded - c.V_real) * H * 2, stream);
        if (e != cudaSuccess) return fail(RLK_ERR_CUDA, std::string("clearing padded dW rows: ") + cudaGetErrorString(e));
    }
    return RLK_OK;
}

}  // namespace rlk
