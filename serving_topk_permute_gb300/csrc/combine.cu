// combine.cu -- unpermute and top-k-weighted reduce (vllm.model_executor.layers.
// fused_moe, DeepGemmExperts.apply: deepgemm_unpermute_and_reduce), plus the
// shared-expert add (DeepGemmMegaMoEExperts.forward: y += shared output) and the
// post-expert RMSNorm with gamma applied verbatim (vllm.models.muse_spark.nvidia.
// mega_moe, finalize_weights / forward_prepared).
//
// One CTA per token; each thread owns 8-column chunks and handles one chunk at a
// time: the k rows' 16-byte pieces of the chunk are loaded in batches of eight
// (independent loads in flight), then z += w[t,j] * y[inv_perm[t,j]] in fp32 in
// ascending j (masked slots skipped), then z += shared. Without a norm the chunk is
// rounded to bf16 and stored at once; with the norm z goes to shared memory, the
// CTA reduces sum(z^2), and a second pass writes z * gamma / sqrt(mean(z^2) + eps).
// Gather-reduce in a fixed order: deterministic, no atomics.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int COMBINE_THREADS = 256;
constexpr int COMBINE_BATCH = 8;

__device__ __forceinline__ void acc_bf16x8(float (&acc)[8], const uint4& v, float w) {
    const uint32_t q[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        acc[2 * i] = fmaf(w, __uint_as_float(q[i] << 16), acc[2 * i]);
        acc[2 * i + 1] = fmaf(w, __uint_as_float(q[i] & 0xFFFF0000u), acc[2 * i + 1]);
    }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&v)[8]) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
        w[j] = *reinterpret_cast<uint32_t*>(&b);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

__global__ void __launch_bounds__(COMBINE_THREADS, 4) combine_kernel(const CombineArgs a) {
    const int t = blockIdx.x, tid = threadIdx.x;
    const int nchunks = a.H / 8;
    extern __shared__ float s_z[];  // [H] when normalising
    __shared__ int s_rows[32];
    __shared__ float s_w[32];
    __shared__ float s_red[COMBINE_THREADS / 32];
    // inv_perm and the weights (an input) are complete before this kernel starts: it
    // starts only after the GEMM launch before it has started, and that launch (or the
    // routed GEMMs before the shared expert's) started only after the routed GEMMs' own
    // wait for dispatch. y is read after the wait, which returns once the GEMM launch
    // before this kernel has completed; a shared-expert launch completes only after the
    // routed GEMMs have.
    if (tid < a.k) {
        s_rows[tid] = __ldcg(a.inv + (int64_t)t * a.k + tid);  // from L2: no stale L1 line
        s_w[tid] = __ldcg(a.w + (int64_t)t * a.k + tid);
    }
    grid_dep_wait();  // the GEMMs have written y (and the shared expert ys)
    grid_dep_launch();
    __syncthreads();
    const bool norm = a.gamma != nullptr;
    uint4* orow = reinterpret_cast<uint4*>(a.out + (int64_t)t * a.H);
    float ss = 0.0f;

    for (int c = tid; c < nchunks; c += COMBINE_THREADS) {
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
        // the shared expert's chunk, loaded beside the k rows' (added after them)
        const uint4 vs = a.ys ? reinterpret_cast<const uint4*>(a.ys + (int64_t)t * a.H)[c] : make_uint4(0, 0, 0, 0);
        for (int j0 = 0; j0 < a.k; j0 += COMBINE_BATCH) {
            uint4 v[COMBINE_BATCH];
#pragma unroll
            for (int u = 0; u < COMBINE_BATCH; ++u) {
                const int j = j0 + u;
                const int r = j < a.k ? s_rows[j] : -1;
                v[u] = r >= 0 ? reinterpret_cast<const uint4*>(a.y + (int64_t)r * a.H)[c] : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int u = 0; u < COMBINE_BATCH; ++u) {
                const int j = j0 + u;
                if (j < a.k && s_rows[j] >= 0) acc_bf16x8(acc, v[u], s_w[j]);
            }
        }
        if (a.ys) acc_bf16x8(acc, vs, 1.0f);
        if (!norm) {
            orow[c] = pack_bf16x8(acc);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                s_z[8 * c + j] = acc[j];
                ss = fmaf(acc[j], acc[j], ss);
            }
        }
    }
    if (!norm) return;

#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (tid % 32 == 0) s_red[tid / 32] = ss;
    __syncthreads();
    float tot = 0.0f;
#pragma unroll
    for (int w = 0; w < COMBINE_THREADS / 32; ++w) tot += s_red[w];
    const float scale = 1.0f / sqrtf(tot / (float)a.H + a.eps);
    for (int c = tid; c < nchunks; c += COMBINE_THREADS) {
        const float4 g0 = reinterpret_cast<const float4*>(a.gamma)[2 * c];  // gamma is 256-byte aligned
        const float4 g1 = reinterpret_cast<const float4*>(a.gamma)[2 * c + 1];
        const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = s_z[8 * c + j] * (g[j] * scale);
        orow[c] = pack_bf16x8(v);
    }
}

cudaError_t combine_prepare() {
    return cudaFuncSetAttribute(combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 16384 * 4);
}

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st, bool pdl) {
    const size_t smem = a.gamma ? (size_t)a.H * sizeof(float) : 0;
    LaunchAttrs at(pdl);
    cudaLaunchConfig_t cfg = at.config(dim3(a.T), dim3(COMBINE_THREADS), smem, st);
    return cudaLaunchKernelEx(&cfg, combine_kernel, a);
}

}  // namespace moe
