// combine.cu -- unpermute and top-k-weighted reduce (vllm.model_executor.layers.
// fused_moe, DeepGemmExperts.apply: deepgemm_unpermute_and_reduce), plus the
// shared-expert add (DeepGemmMegaMoEExperts.forward: y += shared output) and the
// post-expert RMSNorm with gamma applied verbatim (vllm.models.muse_spark.nvidia.
// mega_moe, finalize_weights / forward_prepared).
//
// One CTA per token; each thread owns 8-column chunks. For j = 0..k-1 in that
// order, z += w[t,j] * y[inv_perm[t,j]] in fp32 (masked slots skipped), then
// z += shared, then z * gamma / sqrt(mean(z^2) + eps), then one bf16 rounding.
// Gather-reduce in fixed order: deterministic, no atomics.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int COMBINE_THREADS = 256;
constexpr int COMBINE_MAX_CHUNKS = 8;  // H <= 8 * 256 * 8 = 16384

__device__ __forceinline__ void acc_bf16x8(float (&acc)[8], const uint4& v, float w) {
    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(w, __uint_as_float(q[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(w, __uint_as_float(q[i] & 0xFFFF0000u), acc[2 * i + 1]);
    }
}

__global__ void __launch_bounds__(COMBINE_THREADS) combine_kernel(const CombineArgs a) {
    const int t = blockIdx.x, tid = threadIdx.x;
    const int nchunks = a.H / 8;
    __shared__ int s_rows[32];
    __shared__ float s_w[32];
    __shared__ float s_red[COMBINE_THREADS / 32];
    if (tid < a.k) {
        s_rows[tid] = a.inv[(int64_t)t * a.k + tid];
        s_w[tid] = a.w[(int64_t)t * a.k + tid];
    }
    __syncthreads();

    float acc[COMBINE_MAX_CHUNKS][8];
    // chunk-outer, slot-inner: the k row loads of one chunk are independent and can all be
    // in flight; each element is still summed in ascending j
#pragma unroll
    for (int i = 0; i < COMBINE_MAX_CHUNKS; ++i) {
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
        const int c = tid + i * COMBINE_THREADS;
        if (c >= nchunks) continue;
#pragma unroll 4
        for (int j = 0; j < a.k; ++j) {
            const int r = s_rows[j];
            if (r >= 0) acc_bf16x8(acc[i], reinterpret_cast<const uint4*>(a.y + (int64_t)r * a.H)[c], s_w[j]);
        }
    }
    if (a.ys) {
        const uint4* srow = reinterpret_cast<const uint4*>(a.ys + (int64_t)t * a.H);
#pragma unroll
        for (int i = 0; i < COMBINE_MAX_CHUNKS; ++i) {
            const int c = tid + i * COMBINE_THREADS;
            if (c < nchunks) acc_bf16x8(acc[i], srow[c], 1.0f);
        }
    }
    float scale = 1.0f;
    if (a.gamma) {
        float ss = 0.0f;
#pragma unroll
        for (int i = 0; i < COMBINE_MAX_CHUNKS; ++i)
#pragma unroll
            for (int j = 0; j < 8; ++j) ss = fmaf(acc[i][j], acc[i][j], ss);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (tid % 32 == 0) s_red[tid / 32] = ss;
        __syncthreads();
        float tot = 0.0f;
#pragma unroll
        for (int w = 0; w < COMBINE_THREADS / 32; ++w) tot += s_red[w];
        scale = 1.0f / sqrtf(tot / (float)a.H + a.eps);
    }
    uint4* orow = reinterpret_cast<uint4*>(a.out + (int64_t)t * a.H);
#pragma unroll
    for (int i = 0; i < COMBINE_MAX_CHUNKS; ++i) {
        const int c = tid + i * COMBINE_THREADS;
        if (c >= nchunks) continue;
        float g[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) g[j] = a.gamma ? a.gamma[c * 8 + j] * scale : 1.0f;
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 b = __floats2bfloat162_rn(acc[i][2 * j] * g[2 * j], acc[i][2 * j + 1] * g[2 * j + 1]);
            w[j] = *reinterpret_cast<uint32_t*>(&b);
        }
        orow[c] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st) {
    combine_kernel<<<a.T, COMBINE_THREADS, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
