/*
 * Device (CUDA) build of the seeded synthetic-input generator.
 *
 * Same arguments and same bits as synth_host.c; used to fill tensors that
 * are too large to generate on the host and copy (the 20 GB logits of a
 * 65536 x 152576 batch).  Every float step is an explicitly rounded single
 * operation (__fmul_rn, __fadd_rn), so nothing is contracted into an FMA.
 */
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth_core.h"

namespace {

constexpr int kMaxSpikes = 16;

__global__ void logits_kernel(uint16_t* out, int64_t row0, int64_t nrows, int64_t row_stride,
                              int64_t v_padded, int64_t v_real, uint64_t seed, float scale,
                              int32_t nspikes, float spike, int32_t garbage) {
    __shared__ int64_t spikes[kMaxSpikes];
    const uint64_t k_val = syn_key(seed, SYN_STREAM_LOGITS);
    const uint64_t k_spk = syn_key(seed, SYN_STREAM_SPIKES);
    const uint64_t k_gar = syn_key(seed, SYN_STREAM_GARBAGE);
    const int ns = nspikes > kMaxSpikes ? kMaxSpikes : nspikes;
    for (int64_t lr = blockIdx.x; lr < nrows; lr += gridDim.x) {
        const uint64_t r = (uint64_t)(row0 + lr);
        __syncthreads();
        if ((int)threadIdx.x < ns)
            spikes[threadIdx.x] = (int64_t)syn_bounded(
                syn_u64(k_spk, r * (uint64_t)ns + threadIdx.x), (uint64_t)v_real);
        __syncthreads();
        uint16_t* row = out + lr * row_stride;
        for (int64_t c = threadIdx.x; c < row_stride; c += blockDim.x) {
            if (c < v_real) {
                float f = __fmul_rn((float)syn_ih12(k_val, syn_ctr2(r, (uint64_t)c)), scale);
                bool hit = false;
                for (int i = 0; i < ns; ++i) hit |= (spikes[i] == c);
                if (hit) f = __fadd_rn(f, spike);
                row[c] = syn_bf16_rne_bits(__float_as_uint(f));
            } else if (c < v_padded || garbage) {
                row[c] = garbage ? (uint16_t)(syn_u64(k_gar, syn_ctr2(r, (uint64_t)c)) & 0xFFFFu) : 0;
            }
        }
    }
}

__global__ void normal_kernel(uint16_t* out, int64_t row0, int64_t nrows, int64_t cols,
                              uint64_t key, float scale) {
    for (int64_t lr = blockIdx.x; lr < nrows; lr += gridDim.x) {
        const uint64_t r = (uint64_t)(row0 + lr);
        uint16_t* row = out + lr * cols;
        for (int64_t c = threadIdx.x; c < cols; c += blockDim.x) {
            float f = __fmul_rn((float)syn_ih12(key, syn_ctr2(r, (uint64_t)c)), scale);
            row[c] = syn_bf16_rne_bits(__float_as_uint(f));
        }
    }
}

int grid_for(int64_t nrows) {
    int64_t g = nrows < 1 ? 1 : nrows;
    return (int)(g > 65535 ? 65535 : g);
}

}  // namespace

/* Device twin of syn_host_logits; `out` is a device pointer.  Returns a cudaError_t. */
extern "C" int syn_dev_logits(uint16_t* out, int64_t row0, int64_t nrows, int64_t row_stride,
                              int64_t v_padded, int64_t v_real, uint64_t seed, float scale,
                              int32_t nspikes, float spike, int32_t garbage, cudaStream_t stream) {
    if (nrows <= 0) return (int)cudaSuccess;
    logits_kernel<<<grid_for(nrows), 512, 0, stream>>>(out, row0, nrows, row_stride, v_padded, v_real,
                                                      seed, scale, nspikes, spike, garbage);
    return (int)cudaGetLastError();
}

/* Device twin of syn_host_normal_bf16; `out` is a device pointer.  Returns a cudaError_t. */
extern "C" int syn_dev_normal_bf16(uint16_t* out, int64_t row0, int64_t nrows, int64_t cols,
                                   uint64_t seed, uint32_t stream_id, float scale, cudaStream_t stream) {
    if (nrows <= 0) return (int)cudaSuccess;
    normal_kernel<<<grid_for(nrows), 512, 0, stream>>>(out, row0, nrows, cols,
                                                      syn_key(seed, stream_id), scale);
    return (int)cudaGetLastError();
}
