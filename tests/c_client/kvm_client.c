/*
 * A plain C client of libkvm: one recall step (Mean-K build, Eq. (10) scoring
 * and selection, view assembly) through the C ABI alone, with device memory
 * from cudaMalloc.  Used by tests/test_gpu_c_client.py, which writes the
 * inputs, runs this program and checks its outputs against the CPU oracle.
 *
 * usage: kvm_client DIR L G H D THETA N MQ S W V
 * DIR holds float32 inputs kpages.bin [N][L][G][32][D], v.bin (same) and
 * q.bin [L][MQ][H][D]; the program writes index.bin [L][G][N][D], raw.bin,
 * scores.bin [N], sel.bin int32 [V], pool_k.bin and pool_v.bin [V][L][G][32][D].
 */
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "kvm.h"

#define CK(x)                                                                   \
    do {                                                                        \
        cudaError_t e_ = (x);                                                   \
        if (e_ != cudaSuccess) {                                                \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));            \
            exit(2);                                                            \
        }                                                                       \
    } while (0)
#define KV(x)                                                                   \
    do {                                                                        \
        kvm_status s_ = (x);                                                    \
        if (s_ != KVM_OK) {                                                     \
            fprintf(stderr, "%s: %s (%s)\n", #x, kvm_status_string(s_),         \
                    kvm_last_error());                                          \
            exit(3);                                                            \
        }                                                                       \
    } while (0)

static void *load(const char *dir, const char *name, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    FILE *f = fopen(path, "rb");
    if (!f) { perror(path); exit(4); }
    void *h = malloc(bytes);
    if (fread(h, 1, bytes, f) != bytes) { fprintf(stderr, "%s: short read\n", path); exit(4); }
    fclose(f);
    void *d = NULL;
    CK(cudaMalloc(&d, bytes));
    CK(cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice));
    free(h);
    return d;
}

static void save(const char *dir, const char *name, const void *d, size_t bytes) {
    char path[4096];
    snprintf(path, sizeof path, "%s/%s", dir, name);
    void *h = malloc(bytes);
    CK(cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost));
    FILE *f = fopen(path, "wb");
    if (!f || fwrite(h, 1, bytes, f) != bytes) { perror(path); exit(5); }
    fclose(f);
    free(h);
}

int main(int argc, char **argv) {
    if (argc != 12) {
        fprintf(stderr, "usage: %s DIR L G H D THETA N MQ S W V\n", argv[0]);
        return 1;
    }
    const char *dir = argv[1];
    const int L = atoi(argv[2]), G = atoi(argv[3]), H = atoi(argv[4]), D = atoi(argv[5]);
    const double theta = atof(argv[6]);
    const int N = atoi(argv[7]), MQ = atoi(argv[8]), S = atoi(argv[9]), W = atoi(argv[10]);
    const int V = atoi(argv[11]);

    kvm_config cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.n_layers = L;
    cfg.n_kv_heads = G;
    cfg.n_q_heads = H;
    cfg.head_dim = D;
    cfg.block_tokens = 32;
    cfg.rope_theta = theta;
    cfg.kv_dtype = cfg.index_dtype = cfg.q_dtype = KVM_F32;
    cfg.sink_blocks = S;
    cfg.recent_blocks = W;
    cfg.view_blocks = V;
    cfg.max_queries = MQ;
    cfg.max_blocks = N;
    cfg.max_positions = 32 * (int64_t)(N > V ? N : V);
    cfg.tile_blocks = 1024;
    cfg.pool_pages = V;
    cfg.index_location = KVM_DEVICE;
    cfg.repo_location = KVM_DEVICE;
    cfg.h2d_batch_blocks = 64;
    cfg.h2d_mode = 1;
    cfg.host_tier_lambda = 0.5;

    const size_t blk = (size_t)L * G * 32 * D * sizeof(float);
    const size_t idx_bytes = (size_t)L * G * N * D * sizeof(float);
    void *kp = load(dir, "kpages.bin", N * blk);
    void *v = load(dir, "v.bin", N * blk);
    void *q = load(dir, "q.bin", (size_t)L * MQ * H * D * sizeof(float));

    const size_t ws_bytes = kvm_workspace_bytes(&cfg);
    if (ws_bytes == 0) { fprintf(stderr, "invalid config\n"); return 6; }
    void *ws = NULL, *index = NULL, *raw = NULL, *scores = NULL, *sel = NULL;
    void *pool_k = NULL, *pool_v = NULL;
    CK(cudaMalloc(&ws, ws_bytes));               /* 256-byte aligned */
    CK(cudaMalloc(&index, idx_bytes));
    CK(cudaMalloc(&raw, N * blk));
    CK(cudaMalloc(&scores, (size_t)N * sizeof(float)));
    CK(cudaMalloc(&sel, (size_t)V * sizeof(int32_t)));
    CK(cudaMalloc(&pool_k, V * blk));
    CK(cudaMalloc(&pool_v, V * blk));
    cudaStream_t st;
    CK(cudaStreamCreate(&st));

    kvm_ctx *ctx = NULL;
    KV(kvm_create(&cfg, ws, ws_bytes, st, &ctx));
    KV(kvm_build_index(ctx, kp, 0, N, index, raw, st));
    int32_t n_sel = 0;
    KV(kvm_score_select(ctx, q, MQ, index, N, (float *)scores, (int32_t *)sel, &n_sel, st));
    KV(kvm_assemble_view(ctx, (const int32_t *)sel, NULL, n_sel, raw, v, pool_k, pool_v, st));
    KV(kvm_sync(ctx, st));

    save(dir, "index.bin", index, idx_bytes);
    save(dir, "raw.bin", raw, N * blk);
    save(dir, "scores.bin", scores, (size_t)N * sizeof(float));
    save(dir, "sel.bin", sel, (size_t)n_sel * sizeof(int32_t));
    save(dir, "pool_k.bin", pool_k, (size_t)n_sel * blk);
    save(dir, "pool_v.bin", pool_v, (size_t)n_sel * blk);
    KV(kvm_destroy(ctx));
    CK(cudaStreamDestroy(st));
    cudaFree(ws); cudaFree(index); cudaFree(raw); cudaFree(scores); cudaFree(sel);
    cudaFree(pool_k); cudaFree(pool_v); cudaFree(kp); cudaFree(v); cudaFree(q);
    printf("ok %d\n", n_sel);
    return 0;
}
