/*
 * c_abi_step.c -- drives libzero1.so from plain C, with no Python or torch.
 *
 * Usage:
 *   c_abi_step plan                      host only: prints the shard plan of a fixed list
 *   c_abi_step step <out.bin>            on a GPU: one local-shard step (fused accumulate +
 *                                        norm, then clip + AdamW + bf16 copy) on deterministic
 *                                        inputs; writes grad, master, m, v (fp32 arenas) and
 *                                        the bf16 copy (uint16) to out.bin, then the norm record
 *   c_abi_step list <out.bin>            the same step through the tensor-list calls, one
 *                                        cudaMalloc per tensor shard; out.bin has the same
 *                                        format (each shard written at its arena offset)
 *   c_abi_step onecall <out.bin>         the same step as one zero1_local_step call
 *
 * Inputs are a fixed function of the element index, so a test can rebuild them.
 * Test infrastructure: it checks that the C ABI is usable as declared.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "zero1.h"

#define N_TENSORS 5
static const int64_t NUMELS[N_TENSORS] = {1000, 7, 4096, 33, 16385};
static const uint8_t NO_DECAY[N_TENSORS] = {0, 1, 0, 1, 0};
#define DP_SIZE 3
#define DP_RANK 1

static int check(int rc, const char* what) {
    if (rc != ZERO1_OK) {
        fprintf(stderr, "%s: %s %s\n", what, zero1_strerror(rc), zero1_last_cuda_error());
        exit(2);
    }
    return rc;
}

static int check_cuda(cudaError_t e, const char* what) {
    if (e != cudaSuccess) {
        fprintf(stderr, "%s: %s\n", what, cudaGetErrorString(e));
        exit(3);
    }
    return 0;
}

/* deterministic inputs: element j of the arena (padding stays 0) */
static uint16_t grad_bits(int64_t j) { return (uint16_t)(0x3a00u + (uint16_t)((j * 37) % 512) - 256u + ((j & 1) ? 0x8000u : 0u)); }
static float master_val(int64_t j) { return (float)((j * 13) % 200 - 100) * 1e-4f; }

/* The step through the tensor-list calls: each quantity of each tensor is its own
 * allocation; h_g / h_p hold the inputs in arena layout. */
static int run_list(const zero1_plan* plan, const uint16_t* h_g, const float* h_p, int64_t n, const char* out) {
    enum { GRAD, MASTER, EXP_AVG, EXP_AVG_SQ, WEIGHT, MICRO, NQ };
    void* bufs[NQ][N_TENSORS];
    const int elem[NQ] = {4, 4, 4, 4, 2, 2};
    int64_t cnt[N_TENSORS], off[N_TENSORS];
    for (int32_t i = 0; i < N_TENSORS; ++i) {
        check(zero1_plan_tensor(plan, i, NULL, &cnt[i], &off[i]), "zero1_plan_tensor");
        for (int q = 0; q < NQ; ++q) {
            bufs[q][i] = NULL;
            if (cnt[i] == 0) continue;
            check_cuda(cudaMalloc(&bufs[q][i], (size_t)cnt[i] * elem[q]), "cudaMalloc");
            check_cuda(cudaMemset(bufs[q][i], 0, (size_t)cnt[i] * elem[q]), "memset");
        }
        if (cnt[i]) {
            check_cuda(cudaMemcpy(bufs[MICRO][i], h_g + off[i], cnt[i] * 2, cudaMemcpyHostToDevice), "H2D");
            check_cuda(cudaMemcpy(bufs[MASTER][i], h_p + off[i], cnt[i] * 4, cudaMemcpyHostToDevice), "H2D");
        }
    }
    cudaStream_t stream;
    check_cuda(cudaStreamCreate(&stream), "stream");
    void* d_lists[NQ];
    for (int q = 0; q < NQ; ++q) {
        check_cuda(cudaMalloc(&d_lists[q], N_TENSORS * sizeof(void*)), "cudaMalloc");
        check(zero1_list_ptrs_upload(plan, (const void* const*)bufs[q], 1, elem[q], d_lists[q],
                                     N_TENSORS * sizeof(void*), stream), "zero1_list_ptrs_upload");
    }
    const size_t tb = zero1_list_table_bytes(plan), wb = zero1_list_workspace_bytes(plan);
    void *d_table, *d_ws;
    zero1_norm_out* d_norm;
    check_cuda(cudaMalloc(&d_table, tb ? tb : 16), "cudaMalloc");
    check_cuda(cudaMalloc(&d_ws, wb ? wb : 16), "cudaMalloc");
    check_cuda(cudaMalloc((void**)&d_norm, 32), "cudaMalloc");
    check(zero1_list_table_upload(plan, d_table, tb, stream), "zero1_list_table_upload");
    zero1_hparams hp = {3e-4, 0.9, 0.95, 1e-8, 0.1, 1.0};
    check(zero1_list_accumulate_norm(plan, d_table, (float* const*)d_lists[GRAD], (const uint16_t* const*)d_lists[MICRO],
                                     1, 1, 1.0, 0.0, d_ws, wb, d_norm, stream), "zero1_list_accumulate_norm");
    check(zero1_list_step(plan, d_table, (float* const*)d_lists[MASTER], (float* const*)d_lists[EXP_AVG],
                          (float* const*)d_lists[EXP_AVG_SQ], (const float* const*)d_lists[GRAD],
                          (uint16_t* const*)d_lists[WEIGHT], &hp, 1, d_norm, stream), "zero1_list_step");
    zero1_norm_out rec;
    check(zero1_read_norm(d_norm, stream, &rec), "zero1_read_norm");

    /* back to arena layout (padding zero), in the format of the arena mode */
    float* h_out = calloc((size_t)n, 4);
    uint16_t* h_w = calloc((size_t)n, 2);
    FILE* f = fopen(out, "wb");
    if (!f) return 4;
    const int order[4] = {GRAD, MASTER, EXP_AVG, EXP_AVG_SQ};
    for (int a = 0; a < 4; ++a) {
        memset(h_out, 0, (size_t)n * 4);
        for (int32_t i = 0; i < N_TENSORS; ++i)
            if (cnt[i])
                check_cuda(cudaMemcpy(h_out + off[i], bufs[order[a]][i], cnt[i] * 4, cudaMemcpyDeviceToHost), "D2H");
        fwrite(h_out, 4, (size_t)n, f);
    }
    for (int32_t i = 0; i < N_TENSORS; ++i)
        if (cnt[i]) check_cuda(cudaMemcpy(h_w + off[i], bufs[WEIGHT][i], cnt[i] * 2, cudaMemcpyDeviceToHost), "D2H");
    fwrite(h_w, 2, (size_t)n, f);
    fwrite(&rec, sizeof rec, 1, f);
    fclose(f);
    printf("ok list sumsq %.17g norm %.17g status %d partials %d\n", rec.sumsq, rec.norm, rec.status, rec.n_partials);
    for (int q = 0; q < NQ; ++q) {
        for (int32_t i = 0; i < N_TENSORS; ++i) cudaFree(bufs[q][i]);
        cudaFree(d_lists[q]);
    }
    cudaFree(d_table); cudaFree(d_ws); cudaFree(d_norm);
    cudaStreamDestroy(stream);
    free(h_out); free(h_w);
    return 0;
}

int main(int argc, char** argv) {
    if (argc < 2) {
        fprintf(stderr, "usage: %s plan | step <out.bin> | list <out.bin> | onecall <out.bin>\n", argv[0]);
        return 1;
    }
    zero1_plan* plan = NULL;
    check(zero1_plan_create(NUMELS, NO_DECAY, N_TENSORS, DP_SIZE, DP_RANK, &plan), "zero1_plan_create");
    const int64_t n = zero1_plan_arena_numel(plan);
    if (strcmp(argv[1], "plan") == 0) {
        printf("total %lld local %lld arena %lld workspace %zu\n", (long long)zero1_plan_total_numel(plan),
               (long long)zero1_plan_local_numel(plan), (long long)n, zero1_workspace_bytes(plan));
        for (int32_t i = 0; i < N_TENSORS; ++i) {
            int64_t s, c, o;
            check(zero1_plan_tensor(plan, i, &s, &c, &o), "zero1_plan_tensor");
            printf("tensor %d start %lld count %lld offset %lld\n", i, (long long)s, (long long)c, (long long)o);
        }
        zero1_plan_destroy(plan);
        return 0;
    }
    const int list_mode = strcmp(argv[1], "list") == 0;
    const int one_call = strcmp(argv[1], "onecall") == 0;
    if ((strcmp(argv[1], "step") != 0 && !list_mode && !one_call) || argc < 3) return 1;

    /* host inputs: the shard elements get values, padding stays zero */
    uint16_t* h_g = calloc((size_t)n, sizeof(uint16_t));
    float* h_p = calloc((size_t)n, sizeof(float));
    for (int32_t i = 0; i < N_TENSORS; ++i) {
        int64_t s, c, o;
        check(zero1_plan_tensor(plan, i, &s, &c, &o), "zero1_plan_tensor");
        for (int64_t k = 0; k < c; ++k) {
            h_g[o + k] = grad_bits(o + k);
            h_p[o + k] = master_val(o + k);
        }
    }
    if (list_mode) {
        int rc = run_list(plan, h_g, h_p, n, argv[2]);
        free(h_g);
        free(h_p);
        zero1_plan_destroy(plan);
        return rc;
    }
    float *d_grad, *d_p, *d_m, *d_v;
    uint16_t *d_w, *d_g;
    void* d_ws;
    zero1_norm_out* d_norm;
    const size_t ws_bytes = zero1_workspace_bytes(plan);
    check_cuda(cudaMalloc((void**)&d_grad, n * 4), "cudaMalloc");
    check_cuda(cudaMalloc((void**)&d_p, n * 4), "cudaMalloc");
    check_cuda(cudaMalloc((void**)&d_m, n * 4), "cudaMalloc");
    check_cuda(cudaMalloc((void**)&d_v, n * 4), "cudaMalloc");
    check_cuda(cudaMalloc((void**)&d_w, n * 2), "cudaMalloc");
    check_cuda(cudaMalloc((void**)&d_g, n * 2), "cudaMalloc");
    check_cuda(cudaMalloc(&d_ws, ws_bytes ? ws_bytes : 16), "cudaMalloc");
    check_cuda(cudaMalloc((void**)&d_norm, 32), "cudaMalloc");
    check_cuda(cudaMemcpy(d_g, h_g, n * 2, cudaMemcpyHostToDevice), "H2D");
    check_cuda(cudaMemcpy(d_p, h_p, n * 4, cudaMemcpyHostToDevice), "H2D");
    check_cuda(cudaMemset(d_m, 0, n * 4), "memset");
    check_cuda(cudaMemset(d_v, 0, n * 4), "memset");
    check_cuda(cudaMemset(d_w, 0, n * 2), "memset");

    cudaStream_t stream;
    check_cuda(cudaStreamCreate(&stream), "stream");
    const uint16_t* micro[1] = {d_g};
    zero1_hparams hp = {3e-4, 0.9, 0.95, 1e-8, 0.1, 1.0};
    if (one_call) {
        check(zero1_local_step(plan, d_grad, micro, 1, 1.0, 0.0, d_ws, ws_bytes, d_norm, d_p, d_m, d_v, d_w, &hp, 1,
                               stream), "zero1_local_step");
    } else {
        check(zero1_accumulate_norm(plan, d_grad, micro, 1, 1, 1.0, 0.0, d_ws, ws_bytes, d_norm, stream),
              "zero1_accumulate_norm");
        check(zero1_step(plan, d_p, d_m, d_v, d_grad, d_w, &hp, 1, d_norm, stream), "zero1_step");
    }
    zero1_norm_out rec;
    check(zero1_read_norm(d_norm, stream, &rec), "zero1_read_norm");

    float* h_out = malloc((size_t)n * 4);
    uint16_t* h_w = malloc((size_t)n * 2);
    FILE* f = fopen(argv[2], "wb");
    if (!f) return 4;
    const float* arenas[4] = {d_grad, d_p, d_m, d_v};
    for (int a = 0; a < 4; ++a) {
        check_cuda(cudaMemcpy(h_out, arenas[a], n * 4, cudaMemcpyDeviceToHost), "D2H");
        fwrite(h_out, 4, (size_t)n, f);
    }
    check_cuda(cudaMemcpy(h_w, d_w, n * 2, cudaMemcpyDeviceToHost), "D2H");
    fwrite(h_w, 2, (size_t)n, f);
    fwrite(&rec, sizeof rec, 1, f);
    fclose(f);
    printf("ok arena %lld sumsq %.17g norm %.17g status %d\n", (long long)n, rec.sumsq, rec.norm, rec.status);

    cudaFree(d_grad); cudaFree(d_p); cudaFree(d_m); cudaFree(d_v); cudaFree(d_w); cudaFree(d_g);
    cudaFree(d_ws); cudaFree(d_norm);
    cudaStreamDestroy(stream);
    free(h_g); free(h_p); free(h_out); free(h_w);
    zero1_plan_destroy(plan);
    return 0;
}
