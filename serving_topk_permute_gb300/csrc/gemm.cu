// gemm.cu -- persistent grouped GEMM on tcgen05 for the two expert GEMMs of the
// MoE layer (vllm.model_executor.layers.fused_moe, DeepGemmExperts.apply:
// m_grouped GEMM over BLOCK_M-aligned contiguous expert segments).
//
// Tiles are 128 rows x BN weight rows, BN = 128 (two accumulator buffers in
// tensor memory, so the epilogue of one tile overlaps the MMAs of the next;
// 6-stage ring) or 256 (one accumulator; 4-stage ring).
// One CTA per SM, 576 threads:
//   warp 0 lane 0  TMA producer: A tile (128 rows x 128 B), B tile (BN weight
//                  rows x 128 B), and for MXFP8 / NVFP4 the stage's scale-factor
//                  atoms, into the shared-memory ring (mbarrier tx counts)
//   warp 1 lane 0  MMA issuer: copies the stage's scale atoms to tensor memory
//                  (tcgen05.cp) and issues four 128xBNxK MMAs per stage
//                  (kind::f16 / kind::mxf8f6f4 / kind::mxf4nvf4 block-scaled),
//                  accumulating in tensor memory; commits free the stage
//   warps 2..17    epilogue: 4 warps per tensor-memory lane quarter, each on a
//                  quarter of the tile's columns; one accumulator row per thread
//                  via tcgen05.ld. A warp copies its share of the accumulator
//                  (at most 64 fp32 per thread) into registers and releases it
//                  before it computes and stores, so its work overlaps the MMAs
//                  of the next tile even with a single accumulator buffer.
//                  L1: alpha, SwiGLU (MegaMoEActivation), requantisation of h to
//                  the L2 input format (bf16 / MXFP8 1x32 UE8M0 / NVFP4 1x16 E4M3
//                  under the scalar L2 input scale). L2: alpha, bf16 row store.
// Tiles (row tile, N tile) are walked row-tile-major and strided over the grid.
// Every wait is bounded (MOE_ERR_TIMEOUT in the error word); a CTA that gives up
// still waits for its own copies and MMAs before freeing tensor memory.
#include "gemm_epilogue.cuh"

namespace moe {

template <int FMT, int BN>
struct GemmCfg {
    static_assert(BN == 128 || BN == 256, "tile width");
    static constexpr int S = fmt_sf_atoms(FMT);
    static constexpr int NB = BN / NBLK;                 // 128-row weight blocks per tile
    static constexpr int NUM_ACC = BN == 128 ? 2 : 1;    // accumulator buffers in tensor memory
    static constexpr int STAGES = BN == 128 ? 6 : 4;
    static constexpr int A_BYTES = BM * BK_BYTES;
    static constexpr int B_BYTES = BN * BK_BYTES;
    static constexpr int SFA_BYTES = S * ATOM_BYTES;
    static constexpr int SFB_BYTES = S * NB * ATOM_BYTES;
    static constexpr uint32_t TX_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    static constexpr int STAGE_BYTES = (TX_BYTES + 1023) / 1024 * 1024;
    static constexpr int ACC_COLS = NUM_ACC * BN;
    static constexpr int SF_COLS = 4 * S * (1 + NB);      // tensor-memory columns of one stage's scale atoms
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
    static_assert(ACC_COLS + STAGES * SF_COLS <= TMEM_COLS, "tensor memory budget");
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(2 * STAGES + 2 * NUM_ACC + 1 <= 28, "barrier area");
};

template <int FMT, bool L1, int BN>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmArgs p) {
    using C = GemmCfg<FMT, BN>;
    constexpr int S = C::S, NB = C::NB, STAGES = C::STAGES, NUM_ACC = C::NUM_ACC;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
    // barriers: full[STAGES], empty[STAGES], tfull[NUM_ACC], tempty[NUM_ACC], drain
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 2 * NUM_ACC + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* never = reinterpret_cast<int*>(tmem_slot + 2);  // stays 0: drains ignore the abort flag

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t tfull0 = bar0 + 8 * (2 * STAGES);
    const uint32_t tempty0 = tfull0 + 8 * NUM_ACC;
    const uint32_t drain_bar = tempty0 + 8 * NUM_ACC;
    const uint64_t tmo = p.timeout_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar0 + 8 * s, 1);             // full[s]
            mbar_init(bar0 + 8 * (STAGES + s), 1);  // empty[s]
        }
        for (int a = 0; a < NUM_ACC; ++a) {
            mbar_init(tfull0 + 8 * a, 1);
            mbar_init(tempty0 + 8 * a, EPI_WARPS);
        }
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
    grid_dep_wait();  // the set-up above overlaps the previous kernel; everything below reads its output
    grid_dep_launch();

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
            int last_parity[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s) last_parity[s] = -1;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                const int mt = tile / p.n_tiles, nt = tile % p.n_tiles;
                const int e = p.tile_expert ? p.tile_expert[mt] : 0;
                for (int ks = 0; ks < p.nks; ++ks) {
                    const uint32_t full = bar0 + 8 * stage, empty = bar0 + 8 * (STAGES + stage);
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
                        const int64_t blk = ((int64_t)e * p.nks + ks) * p.sf_blocks + (int64_t)nt * NB;
                        bulk_load(st + C::A_BYTES + C::B_BYTES + C::SFA_BYTES, p.sfb + blk * S * ATOM_BYTES,
                                  C::SFB_BYTES, full);
                    }
                    last_parity[stage] = (int)phase;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // every load this thread issued lands before the CTA may exit
            for (int s = 0; s < STAGES; ++s)
                if (last_parity[s] >= 0) mbar_wait(bar0 + 8 * s, (uint32_t)last_parity[s], DRAIN_TIMEOUT_NS, never);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, tmo, abort_flag)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int ks = 0; ks < p.nks; ++ks) {
                    const uint32_t full = bar0 + 8 * stage, empty = bar0 + 8 * (STAGES + stage);
                    if (!mbar_wait(full, phase, tmo, abort_flag)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t st = smem_u32(smem + stage * C::STAGE_BYTES);
                    const uint32_t sfa_col = tmem_base + C::ACC_COLS + stage * C::SF_COLS;
                    const uint32_t sfb_col = sfa_col + 4 * S;
                    if constexpr (S > 0) {
                        const uint32_t sfa_smem = st + C::A_BYTES + C::B_BYTES;
#pragma unroll
                        for (int a = 0; a < S; ++a) tc_cp_sf_atom(sfa_col + 4 * a, sf_atom_desc(sfa_smem + a * ATOM_BYTES));
                        // smem holds the weight atoms as [block][s]; tensor memory wants [s][block]
#pragma unroll
                        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                            for (int a = 0; a < S; ++a)
                                tc_cp_sf_atom(sfb_col + 4 * (a * NB + nb),
                                              sf_atom_desc(sfa_smem + C::SFA_BYTES + (nb * S + a) * ATOM_BYTES));
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint64_t ad = kmajor_sw128_desc(st + j * 32);
                        const uint64_t bd = kmajor_sw128_desc(st + C::A_BYTES + j * 32);
                        const uint32_t accumulate = (ks > 0 || j > 0) ? 1u : 0u;
                        if constexpr (FMT == MOE_FMT_BF16)
                            mma_bf16(d_tmem, ad, bd, idesc_bf16(BN), accumulate);
                        else if constexpr (FMT == MOE_FMT_MXFP4)
                            mma_mxf4(d_tmem, ad, bd, idesc_mxf4(BN, 2u * (j & 1)), sfa_col + 4 * (j >> 1),
                                     sfb_col + 4 * NB * (j >> 1), accumulate);
                        else if constexpr (FMT == MOE_FMT_MXFP8)
                            mma_mxf8(d_tmem, ad, bd, idesc_mxf8(BN, j), sfa_col, sfb_col, accumulate);
                        else
                            mma_nvf4(d_tmem, ad, bd, idesc_nvf4(BN), sfa_col + 4 * j, sfb_col + 4 * NB * j,
                                     accumulate);
                    }
                    tc_commit(empty);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit(tfull0 + 8 * acc);
                if (++acc == NUM_ACC) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            // every MMA and copy this thread issued completes before tensor memory is freed
            tc_commit(drain_bar);
            mbar_wait(drain_bar, 0, DRAIN_TIMEOUT_NS, never);
        }
    } else {
        const int q = warp % 4;           // the lane quarter of tensor memory this warp may read
        const int cg = (warp - 2) / 4;    // which quarter of the tile's columns it handles
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            // warp-uniform: every lane leaves together (a lane left behind would block in __syncwarp)
            if (!__all_sync(0xffffffffu, mbar_wait(tfull0 + 8 * acc, acc_phase, tmo, abort_flag))) {
                give_up();
                break;
            }
            tc_fence_after();
            const int mt = tile / p.n_tiles, nt = tile % p.n_tiles;
            const int e = p.tile_expert ? p.tile_expert[mt] : 0;
            const int row = mt * BM + q * 32 + lane;
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16) + acc * BN;
            // hand the accumulator back as soon as it sits in registers
            const uint32_t tempty = tempty0 + 8 * acc;
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty);
            };
            if constexpr (L1)
                epilogue_l1<FMT, BN>(p, tacc, row, nt, e, cg, release);
            else
                epilogue_l2<FMT, BN>(p, tacc, row, nt, e, cg, release);
            if (++acc == NUM_ACC) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
template <int FMT, bool L1, int BN>
static cudaError_t set_attr() {
    return cudaFuncSetAttribute(grouped_gemm_kernel<FMT, L1, BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                GemmCfg<FMT, BN>::SMEM);
}

template <int FMT>
static cudaError_t prepare_fmt() {
    cudaError_t e;
    if ((e = set_attr<FMT, true, 128>()) != cudaSuccess) return e;
    if ((e = set_attr<FMT, false, 128>()) != cudaSuccess) return e;
    if ((e = set_attr<FMT, true, 256>()) != cudaSuccess) return e;
    return set_attr<FMT, false, 256>();
}

cudaError_t gemm_prepare(int fmt) {
    switch (fmt) {
        case MOE_FMT_BF16: return prepare_fmt<MOE_FMT_BF16>();
        case MOE_FMT_MXFP8: return prepare_fmt<MOE_FMT_MXFP8>();
        case MOE_FMT_MXFP4: return prepare_fmt<MOE_FMT_MXFP4>();
        default: return prepare_fmt<MOE_FMT_NVFP4>();
    }
}

template <int FMT, bool L1, int BN>
static cudaError_t launch_t(const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a, int grid,
                            cudaStream_t st, bool pdl) {
    LaunchAttrs at(pdl);
    cudaLaunchConfig_t cfg = at.config(dim3(grid), dim3(GEMM_THREADS), GemmCfg<FMT, BN>::SMEM, st);
    return cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<FMT, L1, BN>, tmA, tmB, a);
}

template <int FMT>
static cudaError_t launch_fmt(bool l1, int bn, const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                              int grid, cudaStream_t st, bool pdl) {
    if (bn == 128)
        return l1 ? launch_t<FMT, true, 128>(tmA, tmB, a, grid, st, pdl)
                  : launch_t<FMT, false, 128>(tmA, tmB, a, grid, st, pdl);
    return l1 ? launch_t<FMT, true, 256>(tmA, tmB, a, grid, st, pdl)
              : launch_t<FMT, false, 256>(tmA, tmB, a, grid, st, pdl);
}

cudaError_t launch_gemm(int fmt, bool l1, int bn, const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                        int grid, cudaStream_t st, bool pdl) {
    if (bn != 128 && bn != 256) return cudaErrorInvalidValue;
    switch (fmt) {
        case MOE_FMT_BF16: return launch_fmt<MOE_FMT_BF16>(l1, bn, tmA, tmB, a, grid, st, pdl);
        case MOE_FMT_MXFP8: return launch_fmt<MOE_FMT_MXFP8>(l1, bn, tmA, tmB, a, grid, st, pdl);
        case MOE_FMT_MXFP4: return launch_fmt<MOE_FMT_MXFP4>(l1, bn, tmA, tmB, a, grid, st, pdl);
        default: return launch_fmt<MOE_FMT_NVFP4>(l1, bn, tmA, tmB, a, grid, st, pdl);
    }
}

}  // namespace moe
