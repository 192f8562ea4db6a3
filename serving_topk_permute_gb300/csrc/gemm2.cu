// gemm2.cu -- the grouped GEMM on CTA pairs (tcgen05 cta_group::2), for expert
// segments long enough to fill 256-row tiles (the prefill shapes and the dense
// shared expert).
//
// A cluster of two CTAs on two SMs computes one 256 x 256 tile: each CTA stages
// its own 128 A rows and one half (128 rows) of the 256 weight rows per K stage
// (32 KB instead of 48 KB, so 5-6 stages fit instead of 4), plus the scale atoms
// its tensor-memory copy needs (its A rows' atoms and both weight halves' atoms).
// Both CTAs' loads are cta_group::2 tensor copies that complete on the leader's
// "full" barrier, on which each producer arrives with its own byte count (the
// follower remotely); so the leader's MMA thread starts a stage as soon as both
// halves have landed. It issues 256x256xK MMAs that read both CTAs' shared memory
// and write each CTA's 128 accumulator rows into its own tensor memory, and
// commits to the barriers of both CTAs at once. The follower's epilogue warps
// report "accumulator read" to the leader. Tiles are walked row-tile-major and
// strided over the clusters. Every pipeline wait is bounded; at the end the
// producers exchange how many stages each issued, so that every issued copy
// lands before either CTA exits, also when one of them gave up.
#include "gemm_epilogue.cuh"

namespace moe {

template <int FMT>
struct Gemm2Cfg {
    static constexpr int S = fmt_sf_atoms(FMT);
    static constexpr int BN = 256;                      // weight rows per pair tile
    static constexpr int NB = BN / NBLK;
    static constexpr int STAGES = FMT == MOE_FMT_NVFP4 ? 5 : 6;  // NVFP4's larger scale atoms leave room for 5
    static constexpr int A_BYTES = BM * BK_BYTES;      // this CTA's 128 rows
    static constexpr int B_BYTES = NBLK * BK_BYTES;    // this CTA's half of the weight rows
    static constexpr int SFA_BYTES = S * ATOM_BYTES;
    static constexpr int SFB_BYTES = S * NB * ATOM_BYTES;  // both halves: each CTA's MMA half needs all N
    static constexpr uint32_t TX_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    static constexpr int STAGE_BYTES = (TX_BYTES + 1023) / 1024 * 1024;
    static constexpr int ACC_COLS = BN;
    static constexpr int SF_COLS = 4 * S * (1 + NB);
    static constexpr int BAR_BYTES = 256;
    static constexpr int SMEM = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
    static_assert(ACC_COLS + STAGES * SF_COLS <= TMEM_COLS, "tensor memory budget");
    static_assert(SMEM <= 232448, "shared memory budget");
};

template <int FMT, bool L1>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    grouped_gemm2_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmSFA, const __grid_constant__ CUtensorMap tmSFB,
                         const GemmArgs p) {
    using C = Gemm2Cfg<FMT>;
    constexpr int S = C::S, NB = C::NB, STAGES = C::STAGES, BN = C::BN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
    // barriers: full[STAGES], empty[STAGES], tfull, tempty, drain, teardown
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * STAGES + 4);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* never = reinterpret_cast<int*>(tmem_slot + 2);
    volatile uint32_t* peer_issued = tmem_slot + 3;  // leader: stages the follower's producer issued

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t tfull_bar = bar0 + 8 * (2 * STAGES);
    const uint32_t tempty_bar = tfull_bar + 8;
    const uint32_t drain_bar = tfull_bar + 16;
    const uint32_t teardown_bar = tfull_bar + 24;
    const uint64_t tmo = p.timeout_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar0 + 8 * s, leader ? 2 : 1);     // full (the leader's counts): both producers arrive
            mbar_init(bar0 + 8 * (STAGES + s), 1);       // empty: the leader's commit
        }
        mbar_init(tfull_bar, 1);
        mbar_init(tempty_bar, leader ? 2 * EPI_WARPS : EPI_WARPS);
        mbar_init(drain_bar, 1);
        mbar_init(teardown_bar, 1);
        *abort_flag = 0;
        *peer_issued = 0;
        *never = 0;
        fence_mbar_init();
        prefetch_tmap(&tmA);
        prefetch_tmap(&tmB);
        if constexpr (C::S > 0) {
            prefetch_tmap(&tmSFA);
            prefetch_tmap(&tmSFB);
        }
    }
    if (warp == 1) {
        tmem_alloc2(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish2();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the peer's barriers exist before anyone arrives on them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    grid_dep_wait();  // the set-up above overlaps the previous kernel; everything below reads its output
    grid_dep_launch();

    const int pair = blockIdx.x / 2, npairs = gridDim.x / 2;
    const int m_tiles = p.m_tiles_dev ? *p.m_tiles_dev : p.m_tiles_host;  // 256-row tiles
    const int total = m_tiles * p.n_tiles;

    auto give_up = [&]() {
        set_error(p.err, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
    };

    if (warp == 0) {
        if (lane == 0) {
            // Both CTAs count their bytes on the leader's full barrier: each arrives on it
            // with its own transaction count (the follower remotely), and its loads
            // complete on it (cta_group::2), so the leader's MMA thread sees a stage
            // as soon as both halves have landed.
            const uint32_t full_cl0 = mapa_shared(bar0, 0);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0;
            bool ok = true;
            for (int tile = pair; ok && tile < total; tile += npairs) {
                const int mt = tile / p.n_tiles, nt = tile % p.n_tiles;
                const int e = p.tile_expert ? p.tile_expert[mt] : 0;
                const int a_tile = 2 * mt + (int)rank;  // this CTA's 128-row tile
                for (int ks = 0; ks < p.nks; ++ks) {
                    const uint32_t empty = bar0 + 8 * (STAGES + stage), full_cl = full_cl0 + 8 * stage;
                    if (!mbar_wait(empty, phase ^ 1, tmo, abort_flag)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    const uint32_t st = smem_u32(smem + stage * C::STAGE_BYTES);
                    if (leader)
                        mbar_arrive_expect_tx(bar0 + 8 * stage, C::TX_BYTES);
                    else
                        mbar_arrive_expect_tx_cluster(full_cl, C::TX_BYTES);
                    tma_load_2d_cg2(st, &tmA, full_cl, ks * BK_BYTES, a_tile * BM);
                    tma_load_3d_cg2(st + C::A_BYTES, &tmB, full_cl, ks * BK_BYTES, nt * BN + (int)rank * NBLK, e);
                    if constexpr (S > 0) {
                        tma_load_2d_cg2(st + C::A_BYTES + C::B_BYTES, &tmSFA, full_cl, 0,
                                        (a_tile * p.nks + ks) * S);
                        tma_load_2d_cg2(st + C::A_BYTES + C::B_BYTES + C::SFA_BYTES, &tmSFB, full_cl, 0,
                                        ((e * p.nks + ks) * p.sf_blocks + nt * NB) * S);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            // Every load either CTA issued lands before the pair may exit. The follower
            // reports its count to the leader; for a stage only one CTA issued (one of
            // them gave up), the leader supplies the missing arrival, so that the stage's
            // phase completes once the issued bytes have landed. A producer can run at
            // most STAGES stages ahead of the other one (a slot is reused only after the
            // MMA consumed it, which needs both arrivals), so each slot is touched once.
            if (!leader) {
                st_cluster_u32(mapa_shared(smem_u32((const void*)peer_issued), 0), issued);
                mbar_arrive_release_cluster(mapa_shared(teardown_bar, 0));
            } else {
                uint32_t other = issued;
                if (mbar_wait_cl(teardown_bar, 0, DRAIN_TIMEOUT_NS, never)) other = *peer_issued;
                const uint32_t lo = min(issued, other), hi = max(issued, other);
                for (uint32_t n = lo; n < hi; ++n) mbar_arrive(bar0 + 8 * (n % STAGES));
                for (uint32_t s = 0; s < (uint32_t)STAGES && s < hi; ++s) {
                    const uint32_t last = s + (hi - 1 - s) / STAGES * STAGES;  // last stage n < hi in slot s
                    mbar_wait(bar0 + 8 * s, (last / STAGES) & 1u, DRAIN_TIMEOUT_NS, never);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            bool issued = false;
            for (int tile = pair; ok && tile < total; tile += npairs) {
                if (!mbar_wait_cl(tempty_bar, acc_phase ^ 1, tmo, abort_flag)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                for (int ks = 0; ks < p.nks; ++ks) {
                    const uint32_t full = bar0 + 8 * stage, empty = bar0 + 8 * (STAGES + stage);
                    if (!mbar_wait_cl(full, phase, tmo, abort_flag)) {
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
                        for (int a = 0; a < S; ++a)
                            tc_cp2_sf_atom(sfa_col + 4 * a, sf_atom_desc(sfa_smem + a * ATOM_BYTES));
                        // shared memory holds the weight atoms as [block][s]; tensor memory wants [s][block]
#pragma unroll
                        for (int nb = 0; nb < NB; ++nb)
#pragma unroll
                            for (int a = 0; a < S; ++a)
                                tc_cp2_sf_atom(sfb_col + 4 * (a * NB + nb),
                                               sf_atom_desc(sfa_smem + C::SFA_BYTES + (nb * S + a) * ATOM_BYTES));
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const uint64_t ad = kmajor_sw128_desc(st + j * 32);
                        const uint64_t bd = kmajor_sw128_desc(st + C::A_BYTES + j * 32);
                        const uint32_t accumulate = (ks > 0 || j > 0) ? 1u : 0u;
                        if constexpr (FMT == MOE_FMT_BF16)
                            mma2_bf16(tmem_base, ad, bd, idesc_m(idesc_bf16(BN), 2 * BM), accumulate);
                        else if constexpr (FMT == MOE_FMT_MXFP4)
                            mma2_mxf4(tmem_base, ad, bd, idesc_m(idesc_mxf4(BN, 2u * (j & 1)), 2 * BM),
                                      sfa_col + 4 * (j >> 1), sfb_col + 4 * NB * (j >> 1), accumulate);
                        else if constexpr (FMT == MOE_FMT_MXFP8)
                            mma2_mxf8(tmem_base, ad, bd, idesc_m(idesc_mxf8(BN, j), 2 * BM), sfa_col, sfb_col,
                                      accumulate);
                        else
                            mma2_nvf4(tmem_base, ad, bd, idesc_m(idesc_nvf4(BN), 2 * BM), sfa_col + 4 * j,
                                      sfb_col + 4 * NB * j, accumulate);
                    }
                    issued = true;
                    tc_commit2_mc(empty, 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit2_mc(tfull_bar, 0x3);
                acc_phase ^= 1;
            }
            // every MMA and copy issued completes before either CTA frees its tensor memory
            if (issued) {
                tc_commit2_mc(drain_bar, 0x1);
                mbar_wait(drain_bar, 0, DRAIN_TIMEOUT_NS, never);
            }
        }
    } else {
        const int q = warp % 4;
        const int cg = (warp - 2) / 4;
        const uint32_t leader_tempty = mapa_shared(tempty_bar, 0);
        uint32_t acc_phase = 0;
        for (int tile = pair; tile < total; tile += npairs) {
            // warp-uniform: every lane leaves together (a lane left behind would block in __syncwarp)
            if (!__all_sync(0xffffffffu, mbar_wait(tfull_bar, acc_phase, tmo, abort_flag))) {
                give_up();
                break;
            }
            tc_fence_after();
            const int mt = tile / p.n_tiles, nt = tile % p.n_tiles;
            const int e = p.tile_expert ? p.tile_expert[mt] : 0;
            const int row = mt * 2 * BM + (int)rank * BM + q * 32 + lane;
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16);
            // hand the accumulator back as soon as it sits in registers
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if (leader)
                        mbar_arrive(tempty_bar);
                    else
                        mbar_arrive_cluster(leader_tempty);
                }
            };
            if constexpr (L1)
                epilogue_l1<FMT, BN>(p, tacc, row, nt, e, cg, release);
            else
                epilogue_l2<FMT, BN>(p, tacc, row, nt, e, cg, release);
            acc_phase ^= 1;
        }
    }
    __syncthreads();
    cluster_sync();  // both CTAs are done with each other's barriers and the MMAs have drained
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc2(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side
template <int FMT, bool L1>
static cudaError_t set_attr2() {
    return cudaFuncSetAttribute(grouped_gemm2_kernel<FMT, L1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Gemm2Cfg<FMT>::SMEM);
}

cudaError_t gemm2_prepare(int fmt) {
    cudaError_t e;
    switch (fmt) {
        case MOE_FMT_BF16:
            if ((e = set_attr2<MOE_FMT_BF16, true>()) != cudaSuccess) return e;
            return set_attr2<MOE_FMT_BF16, false>();
        case MOE_FMT_MXFP8:
            if ((e = set_attr2<MOE_FMT_MXFP8, true>()) != cudaSuccess) return e;
            return set_attr2<MOE_FMT_MXFP8, false>();
        case MOE_FMT_MXFP4:
            if ((e = set_attr2<MOE_FMT_MXFP4, true>()) != cudaSuccess) return e;
            return set_attr2<MOE_FMT_MXFP4, false>();
        default:
            if ((e = set_attr2<MOE_FMT_NVFP4, true>()) != cudaSuccess) return e;
            return set_attr2<MOE_FMT_NVFP4, false>();
    }
}

template <int FMT, bool L1>
static cudaError_t launch2_t(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmSFA,
                             const CUtensorMap& tmSFB, const GemmArgs& a, int grid, cudaStream_t st, bool pdl) {
    LaunchAttrs at(pdl, 2);
    cudaLaunchConfig_t cfg = at.config(dim3(grid), dim3(GEMM_THREADS), Gemm2Cfg<FMT>::SMEM, st);
    return cudaLaunchKernelEx(&cfg, grouped_gemm2_kernel<FMT, L1>, tmA, tmB, tmSFA, tmSFB, a);
}

// grid: an even number of CTAs (pairs); the B tensor map's box is 128 rows (one half)
cudaError_t launch_gemm2(int fmt, bool l1, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmSFA,
                         const CUtensorMap& tmSFB, const GemmArgs& a, int grid, cudaStream_t st, bool pdl) {
    if (grid % 2) return cudaErrorInvalidValue;
    switch (fmt) {
        case MOE_FMT_BF16:
            return l1 ? launch2_t<MOE_FMT_BF16, true>(tmA, tmB, tmSFA, tmSFB, a, grid, st, pdl)
                      : launch2_t<MOE_FMT_BF16, false>(tmA, tmB, tmSFA, tmSFB, a, grid, st, pdl);
        case MOE_FMT_MXFP8:
            return l1 ? launch2_t<MOE_FMT_MXFP8, true>(tmA, tmB, tmSFA, tmSFB, a, grid, st, pdl)
                      : launch2_t<MOE_FMT_MXFP8, false>(tmA, tmB, tmSFA, tmSFB, a, grid, st, pdl);
        case MOE_FMT_MXFP4:
            return l1 ? launch2_t<MOE_FMT_MXFP4, true>(tmA, tmB, tmSFA, tmSFB, a, grid, st, pdl)
                      : launch2_t<MOE_FMT_MXFP4, false>(tmA, tmB, tmSFA, tmSFB, a, grid, st, pdl);
        default:
            return l1 ? launch2_t<MOE_FMT_NVFP4, true>(tmA, tmB, tmSFA, tmSFB, a, grid, st, pdl)
                      : launch2_t<MOE_FMT_NVFP4, false>(tmA, tmB, tmSFA, tmSFB, a, grid, st, pdl);
    }
}

}  // namespace moe
