/*
 * A plain C user of libfp8z1.so: no PyTorch, only the header, the library and
 * the CUDA runtime.  Used by tests/test_c_abi.py.
 *
 *   c_abi_example host            host-only calls (layout, shard ranges, LUT,
 *                                  param-wise split, loss scaler, errors)
 *   c_abi_example gpu <in> <out>  one optimizer step on the device: reads
 *                                  grads and master of a 300x200 weight from
 *                                  <in> (raw float32, grads then master),
 *                                  writes master, scales and FP8 weights to
 *                                  <out> (raw: float32 x 6*16384, float32 x 6,
 *                                  uint8 x 300*200)
 *   c_abi_example graph <in> <out> the same, as three steps (t = 1, 2, 3, the
 *                                  same grads) replayed from one CUDA graph:
 *                                  zero the accumulators, norm, copy of the
 *                                  step scalars from pinned memory, step
 *   c_abi_example graph_patch <in> <out>  the same three steps from one graph
 *                                  of the by-value step, whose scalars are
 *                                  rewritten in the executable graph before
 *                                  each launch (fp8z1_graph_set_step_hp)
 */
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "fp8z1.h"

#define CHECK(x)                                                                   \
    do {                                                                           \
        int st_ = (x);                                                             \
        if (st_ != FP8Z1_OK) {                                                     \
            fprintf(stderr, "%s:%d %s -> %s\n", __FILE__, __LINE__, #x, fp8z1_strerror(st_)); \
            return 1;                                                              \
        }                                                                          \
    } while (0)
#define CUDA(x)                                                                    \
    do {                                                                           \
        if ((x) != cudaSuccess) {                                                  \
            fprintf(stderr, "%s:%d %s failed\n", __FILE__, __LINE__, #x);          \
            return 1;                                                              \
        }                                                                          \
    } while (0)

static int host_part(void)
{
    fp8z1_shape shapes[2] = {{1, 300, 200}, {2, 129, 257}};
    fp8z1_layout* L = NULL;
    CHECK(fp8z1_build_layout(shapes, 2, 2, FP8Z1_LAYOUT_HOST_ONLY, &L));
    int64_t nblk = 0, padded = 0, real = 0;
    CHECK(fp8z1_layout_info(L, &nblk, &padded, &real));
    int64_t b0, b1, c0, c1;
    CHECK(fp8z1_shard_range(L, 0, &b0, &b1));
    CHECK(fp8z1_shard_range(L, 1, &c0, &c1));
    fp8z1_block lut[64];
    CHECK(fp8z1_copy_lut(L, lut, 64));
    int32_t owner[2];
    int64_t buckets[2], tot = 0;
    CHECK(fp8z1_paramwise_split(shapes, 2, 2, owner, buckets, &tot));
    fp8z1_loss_scaler sc = {65536.0f, 0, 0, 1000};
    CHECK(fp8z1_scaler_update(&sc, 0));
    CHECK(fp8z1_scaler_update(&sc, 1));
    CHECK(fp8z1_scaler_update(&sc, 0));
    /* a rejected call: rank out of range */
    int bad = fp8z1_shard_range(L, 2, &b0, &b1);
    printf("nblk %lld padded %lld real %lld r0 %lld %lld r1 %lld %lld\n", (long long)nblk,
           (long long)padded, (long long)real, (long long)b0, (long long)b1, (long long)c0, (long long)c1);
    printf("lut5 %d %d %d %d %d %d\n", lut[5].param, lut[5].expert, lut[5].row_block, lut[5].col_block,
           lut[5].rows_real, lut[5].cols_real);
    printf("split %d %d %lld %lld %lld\n", owner[0], owner[1], (long long)buckets[0], (long long)buckets[1],
           (long long)tot);
    printf("scaler %g %lld\n", sc.scale, (long long)sc.step);
    printf("bad %d %s\n", bad, fp8z1_strerror(bad));
    CHECK(fp8z1_destroy_layout(L));
    return 0;
}

static int gpu_part(const char* in, const char* out, int graph)
{ /* graph: 0 none, 1 device scalars, 2 patched */
    const int64_t R = 300, C = 200, n_real = R * C, nblk = 6, n = nblk * FP8Z1_BLOCK_ELEMS;
    float* h = (float*)malloc(sizeof(float) * 2 * n_real);
    FILE* f = fopen(in, "rb");
    if (!f || fread(h, sizeof(float), 2 * n_real, f) != (size_t)(2 * n_real)) return 1;
    fclose(f);
    fp8z1_shape shape = {1, R, C};
    fp8z1_layout* L = NULL;
    CHECK(fp8z1_build_layout(&shape, 1, 1, 0, &L));
    float *d_grad_rm, *d_master_rm, *d_master, *d_m, *d_v, *d_scales;
    uint8_t* d_fp8_rm;
    double* d_sumsq;
    int32_t* d_found;
    void** d_ptrs;
    CUDA(cudaMalloc((void**)&d_grad_rm, sizeof(float) * n_real));
    CUDA(cudaMalloc((void**)&d_master_rm, sizeof(float) * n_real));
    CUDA(cudaMalloc((void**)&d_master, sizeof(float) * n));
    CUDA(cudaMalloc((void**)&d_m, sizeof(float) * n));
    CUDA(cudaMalloc((void**)&d_v, sizeof(float) * n));
    CUDA(cudaMalloc((void**)&d_scales, sizeof(float) * nblk));
    CUDA(cudaMalloc((void**)&d_fp8_rm, n_real));
    CUDA(cudaMalloc((void**)&d_sumsq, sizeof(double)));
    CUDA(cudaMalloc((void**)&d_found, sizeof(int32_t)));
    CUDA(cudaMalloc((void**)&d_ptrs, 3 * sizeof(void*)));
    CUDA(cudaMemcpy(d_grad_rm, h, sizeof(float) * n_real, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(d_master_rm, h + n_real, sizeof(float) * n_real, cudaMemcpyHostToDevice));
    CUDA(cudaMemset(d_m, 0, sizeof(float) * n));
    CUDA(cudaMemset(d_v, 0, sizeof(float) * n));
    CUDA(cudaMemset(d_sumsq, 0, sizeof(double)));
    CUDA(cudaMemset(d_found, 0, sizeof(int32_t)));
    void* ptrs[3] = {d_master_rm, d_grad_rm, d_fp8_rm};
    CUDA(cudaMemcpy(d_ptrs, ptrs, sizeof ptrs, cudaMemcpyHostToDevice));
    /* init: fold the row-major master; then one fused step */
    CHECK(fp8z1_fold(L, (const void* const*)&d_ptrs[0], d_master, 4, 0, nblk, NULL));
    fp8z1_adamw_hp hp = {1e-3f, 0.9f, 0.95f, 1e-8f, 0.1f, 1.0f, 1024.0f, 1};
    if (!graph) {
        CHECK(fp8z1_fold_norm(L, (const float* const*)&d_ptrs[1], NULL, 0, nblk, d_sumsq, d_found, NULL));
        CHECK(fp8z1_step_fused(L, &hp, NULL, (const float* const*)&d_ptrs[1], d_master, d_m, d_v, NULL,
                               (uint8_t* const*)&d_ptrs[2], d_scales, NULL, NULL, 0, nblk, d_sumsq, d_found,
                               NULL));
    } else if (graph == 2) {
        cudaStream_t st;
        cudaGraph_t g;
        cudaGraphExec_t ge;
        void* nodes[4];
        int32_t n_nodes = 0;
        CUDA(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
        CUDA(cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal));
        CHECK(fp8z1_norm_reset(d_sumsq, d_found, st));
        CHECK(fp8z1_fold_norm(L, (const float* const*)&d_ptrs[1], NULL, 0, nblk, d_sumsq, d_found, st));
        CHECK(fp8z1_step_fused(L, &hp, NULL, (const float* const*)&d_ptrs[1], d_master, d_m, d_v, NULL,
                               (uint8_t* const*)&d_ptrs[2], d_scales, NULL, NULL, 0, nblk, d_sumsq, d_found, st));
        CUDA(cudaStreamEndCapture(st, &g));
        CUDA(cudaGraphInstantiate(&ge, g, 0));
        CHECK(fp8z1_graph_step_nodes(g, nodes, 4, &n_nodes));
        if (n_nodes != 1) return 1;
        for (int64_t t = 1; t <= 3; ++t) {
            hp.step = t;
            CHECK(fp8z1_graph_set_step_hp(ge, nodes, n_nodes, &hp));
            CUDA(cudaGraphLaunch(ge, st));
        }
        CUDA(cudaStreamSynchronize(st));
        CUDA(cudaGraphExecDestroy(ge));
        CUDA(cudaGraphDestroy(g));
        CUDA(cudaStreamDestroy(st));
    } else {
        fp8z1_step_scalars *h_sc, *d_sc;
        cudaStream_t st;
        cudaGraph_t g;
        cudaGraphExec_t ge;
        CUDA(cudaHostAlloc((void**)&h_sc, sizeof *h_sc, cudaHostAllocDefault));
        CUDA(cudaMalloc((void**)&d_sc, sizeof *d_sc));
        CUDA(cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking));
        CHECK(fp8z1_step_scalars_from_hp(&hp, h_sc));
        CUDA(cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal));
        CUDA(cudaMemsetAsync(d_sumsq, 0, sizeof(double), st));
        CUDA(cudaMemsetAsync(d_found, 0, sizeof(int32_t), st));
        CHECK(fp8z1_fold_norm(L, (const float* const*)&d_ptrs[1], NULL, 0, nblk, d_sumsq, d_found, st));
        CHECK(fp8z1_step_fused_dev(L, h_sc, d_sc, NULL, (const float* const*)&d_ptrs[1], d_master, d_m, d_v,
                                   NULL, (uint8_t* const*)&d_ptrs[2], d_scales, NULL, NULL, 0, nblk, d_sumsq,
                                   d_found, st));
        CUDA(cudaStreamEndCapture(st, &g));
        CUDA(cudaGraphInstantiate(&ge, g, 0));
        for (int64_t t = 1; t <= 3; ++t) {
            hp.step = t;
            CHECK(fp8z1_step_scalars_from_hp(&hp, h_sc)); /* the previous replay has finished */
            CUDA(cudaGraphLaunch(ge, st));
            CUDA(cudaStreamSynchronize(st));
        }
        CUDA(cudaGraphExecDestroy(ge));
        CUDA(cudaGraphDestroy(g));
        CUDA(cudaStreamDestroy(st));
        CUDA(cudaFree(d_sc));
        CUDA(cudaFreeHost(h_sc));
    }
    CUDA(cudaDeviceSynchronize());
    float* hm = (float*)malloc(sizeof(float) * n);
    float hs[6];
    uint8_t* hq = (uint8_t*)malloc(n_real);
    CUDA(cudaMemcpy(hm, d_master, sizeof(float) * n, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(hs, d_scales, sizeof hs, cudaMemcpyDeviceToHost));
    CUDA(cudaMemcpy(hq, d_fp8_rm, n_real, cudaMemcpyDeviceToHost));
    f = fopen(out, "wb");
    if (!f) return 1;
    fwrite(hm, sizeof(float), n, f);
    fwrite(hs, sizeof(float), 6, f);
    fwrite(hq, 1, n_real, f);
    fclose(f);
    CHECK(fp8z1_destroy_layout(L));
    printf("gpu ok\n");
    return 0;
}

int main(int argc, char** argv)
{
    if (argc >= 2 && strcmp(argv[1], "host") == 0) return host_part();
    if (argc >= 4 && strcmp(argv[1], "gpu") == 0) return gpu_part(argv[2], argv[3], 0);
    if (argc >= 4 && strcmp(argv[1], "graph") == 0) return gpu_part(argv[2], argv[3], 1);
    if (argc >= 4 && strcmp(argv[1], "graph_patch") == 0) return gpu_part(argv[2], argv[3], 2);
    fprintf(stderr, "usage: %s host | gpu|graph|graph_patch <in> <out>\n", argv[0]);
    return 2;
}
