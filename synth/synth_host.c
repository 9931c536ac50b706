/*
 * Host (CPU) build of the seeded synthetic-input generator.
 *
 * Fills BF16 logit rows, BF16 normal matrices, targets, response masks and
 * per-sequence normals from the counter-based core in synth_core.h.  The
 * CUDA build (synth_dev.cu) produces the same bits for the same arguments;
 * a GPU test checks that on sampled rows.  Compiled with
 * -ffp-contract=off so that no multiply-add is fused.
 */
#include <pthread.h>
#include <stdint.h>
#include <string.h>
#include <unistd.h>

#include "synth_core.h"

static uint32_t f32_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return u;
}

static int pick_threads(int32_t nthreads, int64_t nrows) {
    long n = nthreads > 0 ? nthreads : sysconf(_SC_NPROCESSORS_ONLN);
    if (n < 1) n = 1;
    if (n > 64) n = 64;
    if (n > nrows) n = (long)(nrows > 0 ? nrows : 1);
    return (int)n;
}

/* ---------------------------------------------------------------- logits */

typedef struct {
    uint16_t* out;
    int64_t row0, nrows, row_stride, v_padded, v_real;
    uint64_t seed;
    float scale;
    int32_t nspikes;
    float spike;
    int32_t garbage;
    int64_t r_begin, r_end; /* local row range of one worker */
} logits_job;

static void logits_rows(const logits_job* j) {
    const uint64_t k_val = syn_key(j->seed, SYN_STREAM_LOGITS);
    const uint64_t k_spk = syn_key(j->seed, SYN_STREAM_SPIKES);
    const uint64_t k_gar = syn_key(j->seed, SYN_STREAM_GARBAGE);
    int64_t spikes[16];
    for (int64_t lr = j->r_begin; lr < j->r_end; ++lr) {
        const uint64_t r = (uint64_t)(j->row0 + lr);
        uint16_t* row = j->out + lr * j->row_stride;
        const int ns = j->nspikes > 16 ? 16 : j->nspikes;
        for (int i = 0; i < ns; ++i)
            spikes[i] = (int64_t)syn_bounded(syn_u64(k_spk, r * (uint64_t)ns + (uint64_t)i),
                                             (uint64_t)j->v_real);
        for (int64_t c = 0; c < j->row_stride; ++c) {
            if (c < j->v_real) {
                float f = (float)syn_ih12(k_val, syn_ctr2(r, (uint64_t)c)) * j->scale;
                int hit = 0;
                for (int i = 0; i < ns; ++i) hit |= (spikes[i] == c);
                if (hit) f = f + j->spike;
                row[c] = syn_bf16_rne_bits(f32_bits(f));
            } else if (c < j->v_padded || j->garbage) {
                row[c] = j->garbage ? (uint16_t)(syn_u64(k_gar, syn_ctr2(r, (uint64_t)c)) & 0xFFFFu) : 0;
            }
        }
    }
}

static void* logits_worker(void* arg) {
    logits_rows((const logits_job*)arg);
    return NULL;
}

/*
 * Rows [row0, row0 + nrows) of a [T, row_stride] BF16 logits buffer into
 * out (nrows * row_stride elements).  Columns below v_real: scale * IH12
 * normal, plus `spike` at nspikes uniform columns of the row.  Columns in
 * [v_real, v_padded): random bit patterns when garbage != 0 (NaN, Inf and
 * huge values included), else zero.  Columns in [v_padded, row_stride):
 * random bits when garbage != 0, else left untouched.
 */
void syn_host_logits(uint16_t* out, int64_t row0, int64_t nrows, int64_t row_stride,
                     int64_t v_padded, int64_t v_real, uint64_t seed, float scale,
                     int32_t nspikes, float spike, int32_t garbage, int32_t nthreads) {
    int nt = pick_threads(nthreads, nrows);
    pthread_t th[64];
    logits_job jobs[64];
    for (int t = 0; t < nt; ++t) {
        logits_job j = {out, row0, nrows, row_stride, v_padded, v_real, seed, scale,
                        nspikes, spike, garbage, nrows * t / nt, nrows * (t + 1) / nt};
        jobs[t] = j;
    }
    for (int t = 1; t < nt; ++t) pthread_create(&th[t], NULL, logits_worker, &jobs[t]);
    logits_rows(&jobs[0]);
    for (int t = 1; t < nt; ++t) pthread_join(th[t], NULL);
}

/* ---------------------------------------------------------------- normal */

typedef struct {
    uint16_t* out;
    int64_t row0, cols;
    uint64_t key;
    float scale;
    int64_t r_begin, r_end;
} normal_job;

static void* normal_worker(void* arg) {
    const normal_job* j = (const normal_job*)arg;
    for (int64_t lr = j->r_begin; lr < j->r_end; ++lr) {
        const uint64_t r = (uint64_t)(j->row0 + lr);
        uint16_t* row = j->out + lr * j->cols;
        for (int64_t c = 0; c < j->cols; ++c) {
            float f = (float)syn_ih12(j->key, syn_ctr2(r, (uint64_t)c)) * j->scale;
            row[c] = syn_bf16_rne_bits(f32_bits(f));
        }
    }
    return NULL;
}

/* Rows [row0, row0 + nrows) of a dense [*, cols] BF16 matrix of scale * IH12. */
void syn_host_normal_bf16(uint16_t* out, int64_t row0, int64_t nrows, int64_t cols,
                          uint64_t seed, uint32_t stream, float scale, int32_t nthreads) {
    int nt = pick_threads(nthreads, nrows);
    pthread_t th[64];
    normal_job jobs[64];
    const uint64_t key = syn_key(seed, stream);
    for (int t = 0; t < nt; ++t) {
        normal_job j = {out, row0, cols, key, scale, nrows * t / nt, nrows * (t + 1) / nt};
        jobs[t] = j;
    }
    for (int t = 1; t < nt; ++t) pthread_create(&th[t], NULL, normal_worker, &jobs[t]);
    normal_worker(&jobs[0]);
    for (int t = 1; t < nt; ++t) pthread_join(th[t], NULL);
}

/* ----------------------------------------------------------- small arrays */

/*
 * Targets uniform in [0, v_real).  When ignore_thresh32 > 0, a row whose
 * 32-bit draw is below it (probability ignore_thresh32 / 2^32) holds
 * ignore_index instead.
 */
void syn_host_targets(int64_t* out, int64_t T, int64_t v_real, uint64_t seed,
                      uint64_t ignore_thresh32, int64_t ignore_index) {
    const uint64_t k_t = syn_key(seed, SYN_STREAM_TARGETS);
    const uint64_t k_i = syn_key(seed, SYN_STREAM_IGNORE);
    for (int64_t r = 0; r < T; ++r) {
        out[r] = (int64_t)syn_bounded(syn_u64(k_t, (uint64_t)r), (uint64_t)v_real);
        if (ignore_thresh32 && (syn_u64(k_i, (uint64_t)r) >> 32) < ignore_thresh32) out[r] = ignore_index;
    }
}

/*
 * Response mask of a [batch, seq] rollout: positions [prompt, prompt + L_b)
 * are active, with L_b uniform in [len_min, len_max] and clamped to
 * seq - prompt.  lens (may be NULL) receives L_b.
 */
void syn_host_response_mask(uint8_t* out, int64_t* lens, int64_t batch, int64_t seq,
                            int64_t prompt, int64_t len_min, int64_t len_max, uint64_t seed) {
    const uint64_t k_l = syn_key(seed, SYN_STREAM_RESPONSE_LEN);
    for (int64_t b = 0; b < batch; ++b) {
        int64_t L = len_min + (int64_t)syn_bounded(syn_u64(k_l, (uint64_t)b), (uint64_t)(len_max - len_min + 1));
        if (L > seq - prompt) L = seq - prompt;
        if (L < 0) L = 0;
        if (lens) lens[b] = L;
        for (int64_t p = 0; p < seq; ++p) out[b * seq + p] = (uint8_t)(p >= prompt && p < prompt + L);
    }
}

/* n standard IH12 normals as doubles (exact: integer / 65536). */
void syn_host_normal_f64(double* out, int64_t n, uint64_t seed, uint32_t stream) {
    const uint64_t key = syn_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = (double)syn_ih12(key, (uint64_t)i) / 65536.0;
}
