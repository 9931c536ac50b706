/*
 * A plain C99 program that uses librlk_logp.so through include/rlk_logp.h
 * alone: no Python, no PyTorch, no C++.  It shows that the boundary is a C
 * ABI and is what tests/test_c_abi_consumer.py compiles and runs.
 *
 *   c_abi_consumer host
 *       Host-only calls (no device is touched): contract checks, workspace
 *       size, status strings, a call that fails closed before any launch.
 *       Prints "host ok" and exits 0 when every answer is the documented one.
 *
 *   c_abi_consumer run T V_real V_padded num_tiles virtual_tp in_dir out_dir
 *       (built with -DRLK_WITH_CUDA, linked with the CUDA runtime)
 *       Reads in_dir/{logits,targets,mask,grad}.bin (BF16 bits [T, V_padded],
 *       int64 [T], uint8 [T], float32 [T]), copies them into cudaMalloc'ed
 *       buffers, runs rlk_logp_fwd and the fused rlk_logp_bwd (lse_in NULL)
 *       with validate = 1, and writes out_dir/{logp,lse,logp_fused,
 *       lse_fused,dlogits}.bin.  Exits non-zero on any failed call.
 *
 * The operation is the selected-token log-probability over a tiled
 * vocabulary (PR #289 "[WS2][PR4][Logp] add distributed TP/CP logprob drift
 * report", the typed logprob contract: FP32 (max, sumexp) tile partials
 * merged in fixed global tile order, logp = logit[target] - LSE).
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "rlk_logp.h"

#ifdef RLK_WITH_CUDA
#include <cuda_runtime.h>
#endif

static int expect(const char* what, rlk_status got, rlk_status want) {
    if (got == want) return 0;
    fprintf(stderr, "%s: got %d (%s), want %d\n", what, (int)got, rlk_status_string(got), (int)want);
    return 1;
}

static rlk_logp_contract make_contract(int64_t T, int64_t vr, int64_t vp, int32_t nt, int32_t vtp) {
    rlk_logp_contract c;
    memset(&c, 0, sizeof c);
    c.T = T;
    c.V_real = vr;
    c.V_padded = vp;
    c.row_stride = 0;
    c.num_tiles = nt;
    c.virtual_tp = vtp;
    c.mask_mode = RLK_MASK_EXPLICIT;
    c.validate = 1;
    c.ignore_index = -100;
    return c;
}

static int host_checks(void) {
    int bad = 0;
    rlk_logp_contract c = make_contract(32, 151936, 152576, 64, 8);
    rlk_logp_contract odd = make_contract(32, 151936, 152576, 63, 1);
    rlk_logp_contract tp3 = make_contract(32, 151936, 152576, 64, 3);
    rlk_logp_contract none = make_contract(0, 151936, 152576, 64, 2);
    bad |= expect("valid contract", rlk_logp_check_contract(&c), RLK_OK);
    bad |= expect("63 tiles of 152576", rlk_logp_check_contract(&odd), RLK_ERR_NON_TILEABLE);
    bad |= expect("virtual_tp 3", rlk_logp_check_contract(&tp3), RLK_ERR_UNSUPPORTED);
    bad |= expect("NULL contract", rlk_logp_check_contract(NULL), RLK_ERR_INVALID_ARG);
    if (rlk_logp_workspace_size(&c) < 4 || rlk_logp_workspace_size(&odd) != 0) {
        fprintf(stderr, "workspace sizes: %zu %zu\n", rlk_logp_workspace_size(&c), rlk_logp_workspace_size(&odd));
        bad = 1;
    }
    /* missing logits: rejected on the host with a reason, before any CUDA call */
    bad |= expect("fwd without logits", rlk_logp_fwd(&c, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL),
                  RLK_ERR_INVALID_ARG);
    if (strlen(rlk_last_error_message()) == 0) {
        fprintf(stderr, "no error message\n");
        bad = 1;
    }
    /* an empty batch is a no-op */
    bad |= expect("empty batch", rlk_logp_fwd(&none, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL), RLK_OK);
    for (int s = RLK_OK; s <= RLK_ERR_CUDA; ++s) {
        const char* str = rlk_status_string((rlk_status)s);
        if (!str || !*str) {
            fprintf(stderr, "status %d has no string\n", s);
            bad = 1;
        }
    }
    if (!bad) printf("host ok\n");
    return bad;
}

#ifdef RLK_WITH_CUDA
static void* read_file(const char* dir, const char* name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "rb");
    if (!f) return NULL;
    void* buf = malloc(bytes ? bytes : 1);
    const size_t got = buf ? fread(buf, 1, bytes, f) : 0;
    fclose(f);
    if (got != bytes) {
        free(buf);
        return NULL;
    }
    return buf;
}

static int write_file(const char* dir, const char* name, const void* buf, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE* f = fopen(path, "wb");
    if (!f) return 1;
    const size_t put = fwrite(buf, 1, bytes, f);
    fclose(f);
    return put != bytes;
}

#define CUDA_OK(call)                                                                        \
    do {                                                                                     \
        cudaError_t e_ = (call);                                                             \
        if (e_ != cudaSuccess) {                                                             \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));                      \
            return 1;                                                                        \
        }                                                                                    \
    } while (0)

static int run(int argc, char** argv) {
    if (argc != 9) {
        fprintf(stderr, "usage: run T V_real V_padded num_tiles virtual_tp in_dir out_dir\n");
        return 2;
    }
    const int64_t T = atoll(argv[2]), vr = atoll(argv[3]), vp = atoll(argv[4]);
    const int32_t nt = atoi(argv[5]), vtp = atoi(argv[6]);
    const char* in = argv[7];
    const char* out = argv[8];
    rlk_logp_contract c = make_contract(T, vr, vp, nt, vtp);
    if (expect("contract", rlk_logp_check_contract(&c), RLK_OK)) return 1;
    const size_t nlog = (size_t)T * (size_t)vp * 2u;
    void* h_logits = read_file(in, "logits.bin", nlog);
    void* h_targets = read_file(in, "targets.bin", (size_t)T * 8u);
    void* h_mask = read_file(in, "mask.bin", (size_t)T);
    void* h_grad = read_file(in, "grad.bin", (size_t)T * 4u);
    if (!h_logits || !h_targets || !h_mask || !h_grad) {
        fprintf(stderr, "cannot read the inputs in %s\n", in);
        return 1;
    }
    void *d_logits, *d_targets, *d_mask, *d_grad, *d_dlogits, *d_ws;
    float *d_logp, *d_lse, *d_logp2, *d_lse2;
    const size_t ws = rlk_logp_workspace_size(&c);
    CUDA_OK(cudaMalloc(&d_logits, nlog));
    CUDA_OK(cudaMalloc(&d_dlogits, nlog));
    CUDA_OK(cudaMalloc(&d_targets, (size_t)T * 8u));
    CUDA_OK(cudaMalloc(&d_mask, (size_t)T));
    CUDA_OK(cudaMalloc(&d_grad, (size_t)T * 4u));
    CUDA_OK(cudaMalloc((void**)&d_logp, (size_t)T * 4u));
    CUDA_OK(cudaMalloc((void**)&d_lse, (size_t)T * 4u));
    CUDA_OK(cudaMalloc((void**)&d_logp2, (size_t)T * 4u));
    CUDA_OK(cudaMalloc((void**)&d_lse2, (size_t)T * 4u));
    CUDA_OK(cudaMalloc(&d_ws, ws));
    CUDA_OK(cudaMemcpy(d_logits, h_logits, nlog, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(d_targets, h_targets, (size_t)T * 8u, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(d_mask, h_mask, (size_t)T, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(d_grad, h_grad, (size_t)T * 4u, cudaMemcpyHostToDevice));

    rlk_status s = rlk_logp_fwd(&c, d_logits, (const int64_t*)d_targets, (const uint8_t*)d_mask, d_logp, d_lse, NULL,
                                d_ws, NULL);
    if (expect("rlk_logp_fwd", s, RLK_OK)) {
        fprintf(stderr, "%s\n", rlk_last_error_message());
        return 1;
    }
    s = rlk_logp_bwd(&c, d_logits, (const int64_t*)d_targets, (const uint8_t*)d_mask, NULL, (const float*)d_grad,
                     d_dlogits, d_logp2, d_lse2, d_ws, NULL);
    if (expect("rlk_logp_bwd (fused)", s, RLK_OK)) {
        fprintf(stderr, "%s\n", rlk_last_error_message());
        return 1;
    }
    CUDA_OK(cudaDeviceSynchronize());
    void* h_out = malloc(nlog > (size_t)T * 4u ? nlog : (size_t)T * 4u);
    if (!h_out) return 1;
    int bad = 0;
    CUDA_OK(cudaMemcpy(h_out, d_logp, (size_t)T * 4u, cudaMemcpyDeviceToHost));
    bad |= write_file(out, "logp.bin", h_out, (size_t)T * 4u);
    CUDA_OK(cudaMemcpy(h_out, d_lse, (size_t)T * 4u, cudaMemcpyDeviceToHost));
    bad |= write_file(out, "lse.bin", h_out, (size_t)T * 4u);
    CUDA_OK(cudaMemcpy(h_out, d_logp2, (size_t)T * 4u, cudaMemcpyDeviceToHost));
    bad |= write_file(out, "logp_fused.bin", h_out, (size_t)T * 4u);
    CUDA_OK(cudaMemcpy(h_out, d_lse2, (size_t)T * 4u, cudaMemcpyDeviceToHost));
    bad |= write_file(out, "lse_fused.bin", h_out, (size_t)T * 4u);
    CUDA_OK(cudaMemcpy(h_out, d_dlogits, nlog, cudaMemcpyDeviceToHost));
    bad |= write_file(out, "dlogits.bin", h_out, nlog);
    free(h_out);
    free(h_logits);
    free(h_targets);
    free(h_mask);
    free(h_grad);
    cudaFree(d_logits);
    cudaFree(d_dlogits);
    cudaFree(d_targets);
    cudaFree(d_mask);
    cudaFree(d_grad);
    cudaFree(d_logp);
    cudaFree(d_lse);
    cudaFree(d_logp2);
    cudaFree(d_lse2);
    cudaFree(d_ws);
    if (bad) fprintf(stderr, "cannot write the outputs in %s\n", out);
    else printf("run ok\n");
    return bad;
}
#endif

int main(int argc, char** argv) {
    if (argc >= 2 && strcmp(argv[1], "host") == 0) return host_checks();
#ifdef RLK_WITH_CUDA
    if (argc >= 2 && strcmp(argv[1], "run") == 0) return run(argc, argv);
#endif
    fprintf(stderr, "usage: %s host | run ...\n", argv[0]);
    return 2;
}
