/*
 * c_abi_forward.c -- one moe_forward driven from plain C through include/moe.h and the
 * CUDA runtime, with no Python and no torch: plan, weight transform, workspace, forward,
 * status. The GPU test test_c_abi_program builds it against libmoe.so, feeds it a seeded
 * case and compares its output with the Python binding's and the oracle's.
 *
 *   c_abi_forward INPUT OUTPUT
 *
 * INPUT (little-endian): "MOEC", int32 E, H, I, k, T, format, then ten blobs, each an
 * int64 byte count followed by the bytes: hidden (bf16 [T, H]), topk_ids (int32 [T, k]),
 * topk_weights (fp32 [T, k]), and the checkpoint-layout routed weights w13, w13_sf, w2,
 * w2_sf, w13_gs, w2_gs, then the NVFP4 L2 input scale (fp32; empty blobs where the
 * format has none). OUTPUT: an int64 byte count and the bf16 output [T, H].
 * Exit status 0 on success; otherwise a message names the call that failed.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "moe.h"

#define NBLOB 10

static int fail_moe(const char* what, int status) {
    fprintf(stderr, "%s failed: %d (%s)\n", what, status, moe_error_string(status));
    return 1;
}

static int fail_cuda(const char* what, cudaError_t e) {
    fprintf(stderr, "%s failed: %s\n", what, cudaGetErrorString(e));
    return 1;
}

/* a host blob copied to a fresh device buffer (NULL for an empty blob) */
static int to_device(const void* host, int64_t bytes, void** dev) {
    *dev = NULL;
    if (bytes == 0) return 0;
    cudaError_t e = cudaMalloc(dev, (size_t)bytes);
    if (e != cudaSuccess) return fail_cuda("cudaMalloc", e);
    e = cudaMemcpy(*dev, host, (size_t)bytes, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return fail_cuda("cudaMemcpy", e);
    return 0;
}

/* a device buffer of the kernel-layout size of one weight tensor (NULL when 0 bytes) */
static int layout_buffer(moe_plan_t plan, int which, void** dev) {
    size_t bytes = 0;
    int st = moe_weight_layout_size(plan, which, &bytes);
    if (st != MOE_OK) return fail_moe("moe_weight_layout_size", st);
    *dev = NULL;
    if (bytes == 0) return 0;
    cudaError_t e = cudaMalloc(dev, bytes);
    if (e != cudaSuccess) return fail_cuda("cudaMalloc", e);
    return 0;
}

int main(int argc, char** argv) {
    if (argc != 3) {
        fprintf(stderr, "usage: %s INPUT OUTPUT\n", argv[0]);
        return 2;
    }
    FILE* f = fopen(argv[1], "rb");
    if (!f) {
        perror("input");
        return 1;
    }
    char magic[4];
    int32_t dims[6];
    if (fread(magic, 1, 4, f) != 4 || memcmp(magic, "MOEC", 4) != 0 || fread(dims, 4, 6, f) != 6) {
        fprintf(stderr, "bad input header\n");
        return 1;
    }
    const int32_t E = dims[0], H = dims[1], I = dims[2], k = dims[3], T = dims[4], fmt = dims[5];
    void* blob[NBLOB];
    int64_t nbytes[NBLOB];
    for (int b = 0; b < NBLOB; ++b) {
        if (fread(&nbytes[b], 8, 1, f) != 1 || nbytes[b] < 0) {
            fprintf(stderr, "bad blob %d\n", b);
            return 1;
        }
        blob[b] = malloc(nbytes[b] > 0 ? (size_t)nbytes[b] : 1);
        if (nbytes[b] > 0 && fread(blob[b], 1, (size_t)nbytes[b], f) != (size_t)nbytes[b]) {
            fprintf(stderr, "short blob %d\n", b);
            return 1;
        }
    }
    fclose(f);

    moe_config_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.num_experts = E;
    cfg.hidden = H;
    cfg.inter = I;
    cfg.top_k = k;
    cfg.max_tokens = T;
    cfg.format = fmt;
    cfg.activation = MOE_ACT_SWIGLU;
    cfg.act_alpha = 1.0f;
    cfg.act_beta = 0.0f;
    cfg.shared_format = MOE_FMT_MXFP8;
    cfg.norm_eps = 1e-6f;
    int st = moe_config_validate(&cfg);
    if (st != MOE_OK) return fail_moe("moe_config_validate", st);
    moe_plan_t plan;
    st = moe_plan(&cfg, &plan);
    if (st != MOE_OK) return fail_moe("moe_plan", st);

    void *d_hidden, *d_ids, *d_w, *d_a2;
    void* d_ck[6];
    if (to_device(blob[0], nbytes[0], &d_hidden) || to_device(blob[1], nbytes[1], &d_ids) ||
        to_device(blob[2], nbytes[2], &d_w))
        return 1;
    for (int b = 0; b < 6; ++b)
        if (to_device(blob[3 + b], nbytes[3 + b], &d_ck[b])) return 1;
    if (to_device(blob[9], nbytes[9], &d_a2)) return 1;

    moe_weights_t src = {d_ck[0], d_ck[1], (float*)d_ck[4], d_ck[2], d_ck[3], (float*)d_ck[5]};
    moe_weights_t dst;
    void* gs13;
    void* gs2;
    if (layout_buffer(plan, MOE_W13, &dst.w13) || layout_buffer(plan, MOE_W13_SF, &dst.w13_sf) ||
        layout_buffer(plan, MOE_W2, &dst.w2) || layout_buffer(plan, MOE_W2_SF, &dst.w2_sf) ||
        layout_buffer(plan, MOE_W13_GS, &gs13) || layout_buffer(plan, MOE_W2_GS, &gs2))
        return 1;
    dst.w13_gs = (float*)gs13;
    dst.w2_gs = (float*)gs2;
    st = moe_transform_weights(plan, &src, &dst, NULL);
    if (st != MOE_OK) return fail_moe("moe_transform_weights", st);

    size_t ws_bytes = 0;
    st = moe_workspace_size(plan, T, &ws_bytes);
    if (st != MOE_OK) return fail_moe("moe_workspace_size", st);
    void* d_ws;
    cudaError_t e = cudaMalloc(&d_ws, ws_bytes);
    if (e != cudaSuccess) return fail_cuda("cudaMalloc", e);
    const size_t out_bytes = (size_t)T * (size_t)H * 2;
    void* d_out;
    e = cudaMalloc(&d_out, out_bytes);
    if (e != cudaSuccess) return fail_cuda("cudaMalloc", e);

    st = moe_forward(plan, T, d_hidden, (const int32_t*)d_ids, (const float*)d_w, &dst, (const float*)d_a2, NULL,
                     NULL, d_out, d_ws, ws_bytes, NULL);
    if (st != MOE_OK) return fail_moe("moe_forward", st);
    int32_t dev_status = -1;
    st = moe_last_status(plan, d_ws, NULL, &dev_status);
    if (st != MOE_OK) return fail_moe("moe_last_status", st);
    if (dev_status != MOE_OK) return fail_moe("device status", dev_status);

    void* out = malloc(out_bytes);
    e = cudaMemcpy(out, d_out, out_bytes, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail_cuda("cudaMemcpy", e);
    FILE* g = fopen(argv[2], "wb");
    if (!g) {
        perror("output");
        return 1;
    }
    const int64_t ob = (int64_t)out_bytes;
    if (fwrite(&ob, 8, 1, g) != 1 || fwrite(out, 1, out_bytes, g) != out_bytes) {
        fprintf(stderr, "write failed\n");
        return 1;
    }
    fclose(g);
    moe_plan_destroy(plan);
    printf("ok: T=%d H=%d E=%d k=%d format=%d\n", T, H, E, k, fmt);
    return 0;
}
