// gemm.cu -- persistent grouped GEMM on tcgen05 for the two expert GEMMs of the
// MoE layer (vllm.model_executor.layers.fused_moe, DeepGemmExperts.apply:
// m_grouped GEMM over BLOCK_M-aligned contiguous expert segments).
//
// One CTA per SM, 192 threads:
//   warp 0 lane 0  TMA producer: A tile (128 rows x 128 B), B tile (256 weight
//                  rows x 128 B), and for MXFP8 / NVFP4 the stage's scale-factor
//                  atoms, into a 4-deep shared-memory ring (mbarrier tx counts)
//   warp 1 lane 0  MMA issuer: copies the stage's scale atoms to tensor memory
//                  (tcgen05.cp) and issues four 128x256xK MMAs per stage
//                  (kind::f16 / kind::mxf8f6f4 / kind::mxf4nvf4 block-scaled),
//                  accumulating in tensor memory; commits free the stage
//   warps 2..5     epilogue: one accumulator row per thread via tcgen05.ld.
//                  L1: alpha, SwiGLU (MegaMoEActivation), requantisation of h to
//                  the L2 input format (bf16 / MXFP8 1x32 UE8M0 / NVFP4 1x16 E4M3
//                  under the scalar L2 input scale). L2: alpha, bf16 row store.
// Tiles (row tile, N tile) are walked row-tile-major and strided over the grid.
// Every wait is bounded (MOE_ERR_TIMEOUT in the error word); a CTA that gives up
// still waits for its own copies and MMAs before freeing tensor memory.
#include "common.cuh"
#include "kernels.h"

namespace moe {

template <int FMT>
struct GemmCfg {
    static constexpr int S = fmt_sf_atoms(FMT);
    static constexpr int A_BYTES = BM * BK_BYTES;
    static constexpr int B_BYTES = BN * BK_BYTES;
    static constexpr int SFA_BYTES = S * ATOM_BYTES;
    static constexpr int SFB_BYTES = S * 2 * ATOM_BYTES;
    static constexpr uint32_t TX_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    static constexpr int STAGE_BYTES = (TX_BYTES + 1023) / 1024 * 1024;
    static constexpr int SF_COLS = 12 * S;  // tensor-memory columns of one stage's scale atoms
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM = NUM_STAGES * STAGE_BYTES + BAR_BYTES + 1024;
    static_assert(ACC_COLS + NUM_STAGES * SF_COLS <= TMEM_COLS, "tensor memory budget");
    static_assert(SMEM <= 232448, "shared memory budget");
};

__device__ __forceinline__ float swiglu_f(float g, float u, const GemmArgs& p) {
    if (p.act_has_clamp) {
        g = fminf(g, p.act_clamp);
        u = fminf(fmaxf(u, -p.act_clamp), p.act_clamp);
    }
    const float sig = 1.0f / (1.0f + expf(-p.act_alpha * g));
    return g * sig * (u + p.act_beta);
}

__device__ __forceinline__ bool row_valid(const GemmArgs& p, int row, int* token) {
    if (p.src) {
        const int s = p.src[row];
        *token = s >= 0 ? s / p.top_k : -1;
        return s >= 0;
    }
    *token = row;
    return row < p.m_valid;
}

template <int FMT>
__device__ __forceinline__ void epilogue_l1(const GemmArgs& p, uint32_t trow, int row, int nt, int e) {
    int t;
    const bool valid = row_valid(p, row, &t);
    float alpha = 1.0f, a2 = 1.0f;
    if constexpr (FMT == MOE_FMT_NVFP4) {
        a2 = *p.a2;
        if (valid) alpha = p.x_scale[t] * p.gscale[e];
    }
#pragma unroll 1
    for (int c = 0; c < BN / 2 / 32; ++c) {
        float g[32], u[32];
        tmem_ld32(trow + c * 32, g);
        tmem_ld32(trow + BN / 2 + c * 32, u);
        tmem_ld_wait();
        if (!valid) continue;
        const int hc = nt * (BN / 2) + c * 32;  // first h column of this chunk
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
}

template <int FMT>
__device__ __forceinline__ void epilogue_l2(const GemmArgs& p, uint32_t trow, int row, int nt, int e) {
    int t;
    const bool valid = row_valid(p, row, &t);
    float alpha = 1.0f;
    if constexpr (FMT == MOE_FMT_NVFP4) alpha = p.gscale[e] * (*p.a2);
#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        float v[32];
        tmem_ld32(trow + c * 32, v);
        tmem_ld_wait();
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

template <int FMT, bool L1>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmArgs p) {
    using C = GemmCfg<FMT>;
    constexpr int S = C::S;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NUM_STAGES * C::STAGE_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * NUM_STAGES + 3);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* never = reinterpret_cast<int*>(tmem_slot + 2);  // stays 0: drains ignore the abort flag

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t tfull_bar = bar0 + 8 * (2 * NUM_STAGES);
    const uint32_t tempty_bar = tfull_bar + 8;
    const uint32_t drain_bar = tfull_bar + 16;
    const uint64_t tmo = p.timeout_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NUM_STAGES; ++s) {
            mbar_init(bar0 + 8 * s, 1);                 // full[s]
            mbar_init(bar0 + 8 * (NUM_STAGES + s), 1);  // empty[s]
        }
        mbar_init(tfull_bar, 1);
        mbar_init(tempty_bar, 4);
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        *never = 0;
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int m_tiles = p.m_tiles_dev ? *p.m_tiles_dev : p.m_tiles_host;
    const int total = m_tiles * p.n_tiles;

    auto give_up = [&]() {
        set_error(p.err, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int last_parity[NUM_STAGES];
#pragma unroll
            for (int s = 0; s < NUM_STAGES; ++s) last_parity[s] = -1;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                const int mt = tile / p.n_tiles, nt = tile % p.n_tiles;
                const int e = p.tile_expert ? p.tile_expert[mt] : 0;
                for (int ks = 0; ks < p.nks; ++ks) {
                    const uint32_t full = bar0 + 8 * stage, empty = bar0 + 8 * (NUM_STAGES + stage);
                    if (!mbar_wait(empty, phase ^ 1, tmo, abort_flag)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    const uint32_t st = smem_u32(smem + stage * C::STAGE_BYTES);
                    mbar_arrive_expect_tx(full, C::TX_BYTES);
                    tma_load_2d(st, &tmA, full, ks * BK_BYTES, mt * BM);
                    tma_load_3d(st + C::A_BYTES, &tmB, full, ks * BK_BYTES, nt * BN, e);
                    if constexpr (S > 0) {
                        bulk_load(st + C::A_BYTES + C::B_BYTES, p.sfa + ((int64_t)mt * p.nks + ks) * C::SFA_BYTES,
                                  C::SFA_BYTES, full);
                        bulk_load(st + C::A_BYTES + C::B_BYTES + C::SFA_BYTES,
                                  p.sfb + (((int64_t)e * p.n_tiles + nt) * p.nks + ks) * C::SFB_BYTES, C::SFB_BYTES,
                                  full);
                    }
                    last_parity[stage] = (int)phase;
                    if (++stage == NUM_STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // every load this thread issued lands before the CTA may exit
            for (int s = 0; s < NUM_STAGES; ++s)
                if (last_parity[s] >= 0) mbar_wait(bar0 + 8 * s, (uint32_t)last_parity[s], tmo, never);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                if (!mbar_wait(tempty_bar, acc_phase ^ 1, tmo, abort_flag)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                for (int ks = 0; ks < p.nks; ++ks) {
                    const uint32_t full = bar0 + 8 * stage, empty = bar0 + 8 * (NUM_STAGES + stage);
                    if (!mbar_wait(full, phase, tmo, abort_flag)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t sf_col = tmem_base + ACC_COLS + stage * C::SF_COLS;
                    if constexpr (S > 0) {
#pragma unroll
                        for (int a = 0; a < 3 * S; ++a)
                            tc_cp_sf_atom(sf_col + 4 * a, sf_atom_desc(st + C::A_BYTES + C::B_BYTES + a * ATOM_BYTES));
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint64_t ad = kmajor_sw128_desc(st + j * 32);
                        const uint64_t bd = kmajor_sw128_desc(st + C::A_BYTES + j * 32);
                        const uint32_t acc = (ks > 0 || j > 0) ? 1u : 0u;
                        if constexpr (FMT == MOE_FMT_BF16)
                            mma_bf16(tmem_base, ad, bd, idesc_bf16(), acc);
                        else if constexpr (FMT == MOE_FMT_MXFP8)
                            mma_mxf8(tmem_base, ad, bd, idesc_mxf8(j), sf_col, sf_col + 4 * S, acc);
                        else
                            mma_nvf4(tmem_base, ad, bd, idesc_nvf4(), sf_col + 4 * j, sf_col + 4 * S + 8 * j, acc);
                    }
                    tc_commit(empty);
                    if (++stage == NUM_STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit(tfull_bar);
                acc_phase ^= 1;
            }
            // every MMA and copy this thread issued completes before tensor memory is freed
            tc_commit(drain_bar);
            mbar_wait(drain_bar, 0, tmo, never);
        }
    } else {
        const int q = warp % 4;  // the lane quarter of tensor memory this warp may read
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            if (!mbar_wait(tfull_bar, acc_phase, tmo, abort_flag)) {
                give_up();
                break;
            }
            tc_fence_after();
            const int mt = tile / p.n_tiles, nt = tile % p.n_tiles;
            const int e = p.tile_expert ? p.tile_expert[mt] : 0;
            const int row = mt * BM + q * 32 + lane;
            const uint32_t trow = tmem_base + ((uint32_t)(q * 32) << 16);
            if constexpr (L1)
                epilogue_l1<FMT>(p, trow, row, nt, e);
            else
                epilogue_l2<FMT>(p, trow, row, nt, e);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar);
            acc_phase ^= 1;
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
template <int FMT, bool L1>
static cudaError_t set_attr() {
    return cudaFuncSetAttribute(grouped_gemm_kernel<FMT, L1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                GemmCfg<FMT>::SMEM);
}

size_t gemm_smem_bytes(int fmt) {
    switch (fmt) {
        case MOE_FMT_BF16: return GemmCfg<MOE_FMT_BF16>::SMEM;
        case MOE_FMT_MXFP8: return GemmCfg<MOE_FMT_MXFP8>::SMEM;
        default: return GemmCfg<MOE_FMT_NVFP4>::SMEM;
    }
}

cudaError_t gemm_prepare(int fmt, bool l1) {
    switch (fmt) {
        case MOE_FMT_BF16: return l1 ? set_attr<MOE_FMT_BF16, true>() : set_attr<MOE_FMT_BF16, false>();
        case MOE_FMT_MXFP8: return l1 ? set_attr<MOE_FMT_MXFP8, true>() : set_attr<MOE_FMT_MXFP8, false>();
        default: return l1 ? set_attr<MOE_FMT_NVFP4, true>() : set_attr<MOE_FMT_NVFP4, false>();
    }
}

template <int FMT, bool L1>
static cudaError_t launch_t(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, int grid,
                            cudaStream_t st) {
    grouped_gemm_kernel<FMT, L1><<<grid, GEMM_THREADS, GemmCfg<FMT>::SMEM, st>>>(tmA, tmB, a);
    return cudaGetLastError();
}

cudaError_t launch_gemm(int fmt, bool l1, const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                        int grid, cudaStream_t st) {
    switch (fmt) {
        case MOE_FMT_BF16:
            return l1 ? launch_t<MOE_FMT_BF16, true>(tmA, tmB, a, grid, st)
                      : launch_t<MOE_FMT_BF16, false>(tmA, tmB, a, grid, st);
        case MOE_FMT_MXFP8:
            return l1 ? launch_t<MOE_FMT_MXFP8, true>(tmA, tmB, a, grid, st)
                      : launch_t<MOE_FMT_MXFP8, false>(tmA, tmB, a, grid, st);
        default:
            return l1 ? launch_t<MOE_FMT_NVFP4, true>(tmA, tmB, a, grid, st)
                      : launch_t<MOE_FMT_NVFP4, false>(tmA, tmB, a, grid, st);
    }
}

}  // namespace moe
