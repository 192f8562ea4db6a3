// gemm_epilogue.cuh -- epilogues shared by the 1-CTA and 2-CTA grouped GEMM kernels:
// one accumulator row per thread, read from tensor memory with tcgen05.ld.
//   L1: alpha (NVFP4: per-token dispatch scale x per-expert w13 global scale),
//       SwiGLU (vllm.model_executor.layers.fused_moe.deep_gemm_mega_moe,
//       MegaMoEActivation: gate * sigmoid(alpha * gate) * (up + beta), clamp first),
//       then requantisation of h to the L2 input format (bf16 / MXFP8 1x32 UE8M0 /
//       NVFP4 1x16 E4M3 under the scalar L2 input scale, fp32 round-to-nearest as in
//       the dispatch quantiser)
//   L2: alpha (NVFP4: w2 global scale x L2 input scale), bf16 row store
#pragma once

#include "common.cuh"
#include "kernels.h"

namespace moe {

__device__ __forceinline__ float swiglu_f(float g, float u, const GemmArgs& p) {
    if (p.act_has_clamp) {
        g = fminf(g, p.act_clamp);
        u = fminf(fmaxf(u, -p.act_clamp), p.act_clamp);
    }
    const float sig = 1.0f / (1.0f + __expf(-p.act_alpha * g));
    return g * sig * (u + p.act_beta);
}

__device__ __forceinline__ bool row_valid(const GemmArgs& p, int row, int* token) {
    if (p.src) {
        const int s = p.src[row];
        *token = s >= 0 ? s / p.top_k : -1;
        return s >= 0;
    }
    *token = row;
    if (p.counts) {
        const int e = row / p.rows_per_expert;
        return row - e * p.rows_per_expert < __ldg(p.counts + e);
    }
    return row < p.m_valid;
}

// Every epilogue first copies its share of the accumulator into registers (64 fp32
// per thread at most), then calls release() -- which hands the accumulator back to
// the MMA issuer -- and only then computes and stores, so that work overlaps the
// next tile's MMAs.

// L1 epilogue, one 32-column chunk of h: chunk k of the tile takes gate columns
// 128 (k/2) + 32 (k%2) and the up columns 64 to their right, and produces h columns
// nt * BN/2 + 32 k .. + 31 (the w13 rows are interleaved by 64 in 128-row blocks).
template <int FMT, int BN, typename Release>
__device__ __forceinline__ void epilogue_l1(const GemmArgs& p, uint32_t tacc, int row, int nt, int e, int cg,
                                            Release release) {
    constexpr int CHUNKS = BN / 64;
    if (cg >= CHUNKS) {  // warp-uniform: this column group has no chunk in narrow tiles
        release();
        return;
    }
    int t;
    const bool valid = row_valid(p, row, &t);
    float alpha = 1.0f, a2 = 1.0f;
    if constexpr (FMT == MOE_FMT_NVFP4) {
        a2 = *p.a2;
        if (valid) alpha = p.x_scale[t] * p.gscale[e];
    }
    const int k = cg;
    const int gcol = 128 * (k / 2) + 32 * (k % 2);
    float g[32], u[32];
    tmem_ld32(tacc + gcol, g);
    tmem_ld32(tacc + gcol + 64, u);
    tmem_ld_wait();
    release();
    if (!valid) return;
    const int hc = nt * (BN / 2) + 32 * k;  // first h column of this chunk
    float h[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) h[i] = swiglu_f(alpha * g[i], alpha * u[i], p);
    if (p.h_debug) {
        float4* dst = reinterpret_cast<float4*>(p.h_debug + (int64_t)row * p.I + hc);
#pragma unroll
        for (int i = 0; i < 8; ++i) dst[i] = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
    }
    if constexpr (FMT == MOE_FMT_BF16) {
        uint4* dst = reinterpret_cast<uint4*>(p.hq + ((int64_t)row * p.I + hc) * 2);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                __nv_bfloat162 b = __floats2bfloat162_rn(h[8 * i + 2 * j], h[8 * i + 2 * j + 1]);
                w[j] = *reinterpret_cast<uint32_t*>(&b);
            }
            dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    } else if constexpr (FMT == MOE_FMT_MXFP8) {
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(h[i]));
        const int ex = ue8m0_exponent(amax);
        uint32_t w[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t lo = cvt_e4m3x2(ldexpf(h[4 * i], -ex), ldexpf(h[4 * i + 1], -ex));
            const uint32_t hi = cvt_e4m3x2(ldexpf(h[4 * i + 2], -ex), ldexpf(h[4 * i + 3], -ex));
            w[i] = lo | (hi << 16);
        }
        uint4* dst = reinterpret_cast<uint4*>(p.hq + (int64_t)row * p.I + hc);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        p.hsf[act_sf_offset(row, hc / 32, 1, p.h_nks)] = (uint8_t)(ex + 127);
    } else if constexpr (FMT == MOE_FMT_MXFP4) {
        // one 1x32 block: UE8M0 exponent with amax <= 6 * 2^ex, E2M1 codes of h * 2^-ex
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(h[i]));
        const int ex = ue8m0_exponent_fp4(amax);
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                word |= cvt_e2m1x2(ldexpf(h[8 * i + 2 * j], -ex), ldexpf(h[8 * i + 2 * j + 1], -ex)) << (8 * j);
            w[i] = word;
        }
        *reinterpret_cast<uint4*>(p.hq + ((int64_t)row * p.I + hc) / 2) = make_uint4(w[0], w[1], w[2], w[3]);
        p.hsf[act_sf_offset(row, hc / 32, 2, p.h_nks)] = (uint8_t)(ex + 127);
    } else {
        const float denom = __fmul_rn(a2, 6.0f);
        uint32_t w[4];
#pragma unroll
        for (int b = 0; b < 2; ++b) {
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(h[16 * b + i]));
            const uint32_t sb = cvt_e4m3x2(__fdiv_rn(amax, denom), 0.0f) & 0xFF;
            const float eff = __fmul_rn(e4m3_to_f32(sb), a2);
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                uint32_t word = 0;
                if (eff > 0.0f) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int idx = 16 * b + 8 * i + 2 * j;
                        word |= cvt_e2m1x2(__fdiv_rn(h[idx], eff), __fdiv_rn(h[idx + 1], eff)) << (8 * j);
                    }
                }
                w[2 * b + i] = word;
            }
            p.hsf[act_sf_offset(row, hc / 16 + b, 4, p.h_nks)] = (uint8_t)sb;
        }
        *reinterpret_cast<uint4*>(p.hq + ((int64_t)row * p.I + hc) / 2) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// L2 epilogue: column group cg (0..3) stores output columns [cg BN/4, (cg+1) BN/4) of the tile
template <int FMT, int BN, typename Release>
__device__ __forceinline__ void epilogue_l2(const GemmArgs& p, uint32_t tacc, int row, int nt, int e, int cg,
                                            Release release) {
    int t;
    const bool valid = row_valid(p, row, &t);
    float alpha = 1.0f;
    if constexpr (FMT == MOE_FMT_NVFP4) alpha = p.gscale[e] * (*p.a2);
    constexpr int PER = BN / 128;  // 32-column chunks per group
    float vv[PER][32];
#pragma unroll
    for (int c = 0; c < PER; ++c) tmem_ld32(tacc + (PER * cg + c) * 32, vv[c]);
    tmem_ld_wait();
    release();
#pragma unroll
    for (int cc = 0; cc < PER; ++cc) {
        const float(&v)[32] = vv[cc];
        const int c = PER * cg + cc;
        const int col = nt * BN + c * 32;
        if (!valid || col >= p.N) continue;
        uint4* dst = reinterpret_cast<uint4*>(p.y + (int64_t)row * p.ldy + col);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                __nv_bfloat162 b = __floats2bfloat162_rn(alpha * v[8 * i + 2 * j], alpha * v[8 * i + 2 * j + 1]);
                w[j] = *reinterpret_cast<uint32_t*>(&b);
            }
            dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

}  // namespace moe
