/*
 * Seeded synthetic-input generator: the counter-based core shared by the host
 * (synth_host.c) and device (synth_dev.cu) builds of this module.
 *
 * This header holds no log-probability arithmetic.  It only turns
 * (seed, stream, counter) triples into bits, so that every element of a
 * synthetic tensor can be regenerated independently and identically on the
 * CPU and on the GPU.
 *
 *   * Hash: the splitmix64 output finaliser (Steele, Lea and Flood,
 *     "Fast splittable pseudorandom number generators", OOPSLA 2014), applied
 *     to key ^ (counter * golden-ratio constant).  Both maps are bijections on
 *     64-bit words, so distinct counters give distinct outputs.
 *   * Bounded integers: Lemire's multiply-shift on the high 32 bits.
 *   * Approximate normals: the Irwin-Hall sum of twelve uniform 16-bit
 *     integers, centred.  The sum has mean 0 and variance 65536^2 - 1, so
 *     s / 65536 has unit variance and support of +-6 sigma.  Everything up to
 *     the single float multiply by the scale is exact integer arithmetic, so
 *     host and device produce the same bits without any transcendental
 *     function.
 *   * BF16: round-to-nearest-even on the float's bit pattern.
 *
 * Every float operation here is one IEEE operation with an explicit rounding
 * (no contraction), which is what makes the two builds bit-identical.
 */
#ifndef SYNTH_CORE_H
#define SYNTH_CORE_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYN_FN __host__ __device__ static inline
#else
#define SYN_FN static inline
#endif

#define SYN_GOLDEN 0x9E3779B97F4A7C15ULL

/* Streams: one per kind of draw, so that tensors never share counters. */
enum {
    SYN_STREAM_LOGITS = 1,
    SYN_STREAM_SPIKES = 2,
    SYN_STREAM_GARBAGE = 3,
    SYN_STREAM_TARGETS = 4,
    SYN_STREAM_IGNORE = 5,
    SYN_STREAM_RESPONSE_LEN = 6,
    SYN_STREAM_ADVANTAGE = 7,
    SYN_STREAM_HIDDEN = 8,
    SYN_STREAM_WEIGHT = 9,
    SYN_STREAM_USER = 16
};

SYN_FN uint64_t syn_mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

SYN_FN uint64_t syn_key(uint64_t seed, uint64_t stream) {
    return syn_mix64(seed * SYN_GOLDEN + stream * 0xD1B54A32D192ED03ULL + 0x632BE59BD9B4E019ULL);
}

SYN_FN uint64_t syn_u64(uint64_t key, uint64_t ctr) {
    return syn_mix64(key ^ (ctr * SYN_GOLDEN));
}

/* Uniform integer in [0, n) for n < 2^32 (multiply-shift on the high word). */
SYN_FN uint64_t syn_bounded(uint64_t u, uint64_t n) {
    return ((u >> 32) * n) >> 32;
}

/* Centred Irwin-Hall(12) integer in [-393210, 393210]; 393210 = 12 * 65535 / 2. */
SYN_FN int32_t syn_ih12(uint64_t key, uint64_t ctr) {
    int64_t s = 0;
    for (int j = 0; j < 3; ++j) {
        uint64_t u = syn_u64(key, ctr * 3u + (uint64_t)j);
        s += (int64_t)(u & 0xFFFFu) + (int64_t)((u >> 16) & 0xFFFFu) +
             (int64_t)((u >> 32) & 0xFFFFu) + (int64_t)(u >> 48);
    }
    return (int32_t)(s - 393210);
}

/* Counter of element (row, col): rows below 2^30, columns below 2^32. */
SYN_FN uint64_t syn_ctr2(uint64_t row, uint64_t col) {
    return (row << 32) | col;
}

/* IEEE float -> BF16 bits, round to nearest even (NaN stays a quiet NaN). */
SYN_FN uint16_t syn_bf16_rne_bits(uint32_t u) {
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

#endif /* SYNTH_CORE_H */
