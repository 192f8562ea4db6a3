// gemm_fused.cu -- both expert GEMMs of the MoE layer in one persistent kernel
// (vllm.model_executor.layers.fused_moe, DeepGemmExperts.apply: GEMM1 -> activation
// -> quant -> GEMM2 over BLOCK_M-aligned expert segments; the pages run them in one
// launch, vllm.model_executor.layers.fused_moe.deep_gemm_mega_moe, module docstring).
//
// The tile list is every L1 tile (row tile x 256 w13 rows) followed by every L2 tile
// (row tile x 256 w2 rows), the row tiles of each phase in the order interleave_tile
// gives (both ends of the expert order, see there). CTAs take tiles in that order
// from a global counter, so the CTAs that finish their L1 work early start L2 tiles
// while others are still on their last L1 tile: the second GEMM has no ramp-up of its
// own and the first no half-empty last round. A row tile with at most 96 used rows
// loads only the 32-row boxes of A that hold them.
//
// An L2 tile of row tile mt reads the L2 input (h codes and scale atoms) of the
// tile's 128 rows, which the epilogues of all L1 tiles of mt write. Each
// epilogue warp publishes its part with a release increment of done[mt] (after a
// fence and a proxy fence), and the producer of an L2 tile waits (bounded) until
// done[mt] counts every warp of every L1 tile of mt, then issues a proxy fence
// before its tensor copies read the rows. A CTA only waits for tiles that running
// CTAs have already taken from the counter, and those never wait on L2 tiles, so
// the waits always end. The routing kernel zeroes the counter and done[] per forward.
//
// Per CTA (one per SM; 576 threads, 704 for NVFP4):
//   warp 0 lane 0  takes tile indices (one fetch ahead), hands each to the other
//                  warps through a 4-entry ring in shared memory, and loads the
//                  tile's A / B / scale-atom stages (TMA tiled + bulk copies)
//   warp 1 lane 0  MMA issuer (tcgen05, 128 x 256 x 32 B per instruction)
//   warps 2..17    epilogue: registers first, then the accumulator is released,
//                  then SwiGLU + requant (L1) or the bf16 row store (L2)
//   warps 18..21   NVFP4: each stage's scale factors, from shared memory into tensor
//                  memory with tcgen05.st (one warp per lane quarter); the other formats'
//                  MMA thread copies its 3 or 6 scale atoms per stage itself (tcgen05.cp)
// Every wait is bounded; a CTA that gives up reports MOE_ERR_TIMEOUT and still waits
// for its own copies and MMAs before freeing tensor memory.
#include "gemm_epilogue.cuh"

namespace moe {

template <int FMT>
struct FusedCfg {
    static constexpr int S = fmt_sf_atoms(FMT);
    static constexpr int BN = 256;
    static constexpr int NB = BN / NBLK;
    static constexpr int STAGES = 4;
    static constexpr int TRING = 4;                     // tile indices in flight between the warps
    static constexpr int PREFETCH_STAGES = 4;           // weight stages of the first tile pulled into L2 early
    static constexpr int A_BYTES = BM * BK_BYTES;
    static constexpr int B_BYTES = BN * BK_BYTES;
    static constexpr int SFA_BYTES = S * ATOM_BYTES;
    static constexpr int SFB_BYTES = S * NB * ATOM_BYTES;
    static constexpr uint32_t TX_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    static constexpr int STAGE_BYTES = (TX_BYTES + 1023) / 1024 * 1024;
    static constexpr int ACC_COLS = BN;
    static constexpr int SF_COLS = 4 * S * (1 + NB);
    // NVFP4 (12 scale-atom copies per stage): four more warps, one per tensor-memory lane
    // quarter, write each stage's scale factors into tensor memory, so that the MMA thread
    // issues only MMAs. (Measured: NVFP4 GEMMs 13% faster; with the 3 or 6 copies per stage
    // of MXFP8 / MXFP4 it was 3-7% slower than the MMA thread's own copies, so those keep them.)
    static constexpr int SF_WARPS = S == 4 ? 4 : 0;
    static constexpr int THREADS = GEMM_THREADS + 32 * SF_WARPS;
    static constexpr int BAR_BYTES = 512;
    static constexpr int SMEM = STAGES * STAGE_BYTES + BAR_BYTES + 1024;
    static_assert(ACC_COLS + STAGES * SF_COLS <= TMEM_COLS, "tensor memory budget");
    static_assert(SMEM <= 232448, "shared memory budget");
    // barriers: full[STAGES], empty[STAGES], tfull, tempty, drain, tile_full[TRING], tile_empty[TRING],
    // sf_full[STAGES]
    static constexpr int NUM_BARS = 3 * STAGES + 3 + 2 * TRING;
    static_assert(NUM_BARS * 8 + (TRING + 4) * 4 <= BAR_BYTES, "barrier area");
};

// Row tiles are taken from both ends of the expert order, TILE_FRONT from the front for
// every TILE_BACK from the back (3, 1: 0, 1, 2, M-1, 3, 4, 5, M-2, ...). Under skewed
// routing the front holds the large experts, whose tiles reuse their weights from L2 and
// keep the tensor cores busy, and the back the small ones, whose tiles stream their
// weights from HBM once; mixing them runs both kinds at the same time instead of one
// phase after the other. (Measured on the Zipf-routed prefill shape: 3:1 beats 1:1, 2:1,
// 4:1 and 6:1 by 1-3%; 1:2 is slower.) A bijection on [0, M): indices 0..M-1 take some
// f front tiles (0 .. f-1) and M - f back tiles (M-1 down to f), which never overlap.
constexpr int TILE_FRONT = 3;
constexpr int TILE_BACK = 1;
__device__ __forceinline__ int interleave_tile(int i, int m) {
    constexpr int G = TILE_FRONT + TILE_BACK;
    const int g = i / G, j = i % G;
    return j < TILE_FRONT ? g * TILE_FRONT + j : m - 1 - (g * TILE_BACK + j - TILE_FRONT);
}

template <int FMT>
__global__ void __launch_bounds__(FusedCfg<FMT>::THREADS, 1)
    fused_mlp_kernel(const __grid_constant__ CUtensorMap tmA1, const __grid_constant__ CUtensorMap tmB1,
                     const __grid_constant__ CUtensorMap tmA2, const __grid_constant__ CUtensorMap tmB2,
                     const __grid_constant__ CUtensorMap tmA1s, const __grid_constant__ CUtensorMap tmA2s,
                     const GemmArgs p1, const GemmArgs p2, const FusedSched fs) {
    using C = FusedCfg<FMT>;
    constexpr int S = C::S, NB = C::NB, STAGES = C::STAGES, BN = C::BN, TRING = C::TRING;
    constexpr int PREFETCH_STAGES = C::PREFETCH_STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + STAGES * C::STAGE_BYTES);
    volatile int* tile_slot = reinterpret_cast<volatile int*>(bars + C::NUM_BARS);  // [TRING]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(const_cast<int*>(tile_slot) + TRING);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* never = reinterpret_cast<int*>(tmem_slot + 2);  // stays 0: drains ignore the abort flag

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t bar0 = smem_u32(bars);
    const uint32_t tfull_bar = bar0 + 8 * (2 * STAGES);
    const uint32_t tempty_bar = tfull_bar + 8;
    const uint32_t drain_bar = tfull_bar + 16;
    const uint32_t tile_full0 = tfull_bar + 24;
    const uint32_t tile_empty0 = tile_full0 + 8 * TRING;
    const uint32_t sf_full0 = tile_empty0 + 8 * TRING;  // a stage's scale factors are in tensor memory
    constexpr bool SFW = C::SF_WARPS > 0;
    const uint64_t tmo = p1.timeout_ns;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar0 + 8 * s, 1);
            mbar_init(bar0 + 8 * (STAGES + s), 1);
        }
        mbar_init(tfull_bar, 1);
        mbar_init(tempty_bar, EPI_WARPS);
        mbar_init(drain_bar, 1);
        for (int r = 0; r < TRING; ++r) {
            mbar_init(tile_full0 + 8 * r, 1);
            mbar_init(tile_empty0 + 8 * r, 1 + EPI_WARPS + C::SF_WARPS);  // the MMA thread, the other warps
        }
        for (int s = 0; s < STAGES; ++s) mbar_init(sf_full0 + 8 * s, SFW ? C::SF_WARPS : 1);
        *abort_flag = 0;
        *never = 0;
        fence_mbar_init();
        prefetch_tmap(&tmA1);
        prefetch_tmap(&tmB1);
        prefetch_tmap(&tmA2);
        prefetch_tmap(&tmB2);
        prefetch_tmap(&tmA1s);
        prefetch_tmap(&tmA2s);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    // What the routing kernel wrote (the row-tile count and experts, the zeroed tile
    // counter) is complete before this kernel starts, even while the kernel just before
    // it (dispatch, or the routed GEMMs before the shared expert) still runs: that kernel
    // lets this one start only after its own grid-dependency wait, so by then routing
    // (and, before the shared expert, dispatch) has finished. So the
    // producer takes its first tile and starts pulling that tile's first weight stages
    // into L2 before the wait, overlapping the previous kernel. (Loads bypass L1.)
    const int m_tiles = p1.m_tiles_dev ? __ldcg(p1.m_tiles_dev) : p1.m_tiles_host;
    const int total1 = m_tiles * p1.n_tiles;
    const int total = total1 + m_tiles * p2.n_tiles;
    const uint32_t done_target = (uint32_t)(EPI_WARPS * p1.n_tiles);
    int first = -1;
    if (warp == 0 && lane == 0) {
        first = (int)atomicAdd(fs.counter, 1u);
        if (first < total1) {
            const int mt = interleave_tile(first / p1.n_tiles, m_tiles), nt = first % p1.n_tiles;
            const int e = p1.tile_expert ? __ldcg(p1.tile_expert + mt) : 0;
            for (int ks = 0; ks < p1.nks && ks < PREFETCH_STAGES; ++ks)
                tma_prefetch_3d(&tmB1, ks * BK_BYTES, nt * BN, e);
        }
    }
    // everything below may read the previous kernel's output; an independent launch reads
    // none of it and waits for that kernel only at its end (a CTA of it becomes resident
    // on an SM only once the previous kernel's CTA there has left, so it fills that
    // kernel's tail)
    if (!fs.independent) grid_dep_wait();
    grid_dep_launch();

    auto give_up = [&]() {
        set_error(p1.err, MOE_ERR_TIMEOUT);
        *abort_flag = 1;
    };
    // tile index -> (phase, row tile, column tile)
    auto decode = [&](int t, bool& l1, int& mt, int& nt) {
        l1 = t < total1;
        const int u = l1 ? t : t - total1;
        const int n = l1 ? p1.n_tiles : p2.n_tiles;
        mt = interleave_tile(u / n, m_tiles);
        nt = u % n;
    };

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int last_parity[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s) last_parity[s] = -1;
            int next = first;
            // A full row tile belongs to an expert with many rows, whose weight tiles the
            // expert's other row tiles read again: keep them in L2. A mostly empty one is
            // (nearly always) an expert's only row tile, whose weights are read once: let them
            // go first, so they do not push the reused weights out. (Measured on the
            // Zipf-routed prefill shape: 1% faster than the default policy for both.)
            const uint64_t pol_reused = make_policy_evict_last(), pol_once = make_policy_evict_first();
            for (int k = 0;; ++k) {
                const int t = next;
                const int r = k % TRING;
                if (!mbar_wait(tile_empty0 + 8 * r, ((k / TRING) & 1) ^ 1, tmo, abort_flag)) {
                    give_up();
                    break;
                }
                tile_slot[r] = t < total ? t : -1;
                mbar_arrive(tile_full0 + 8 * r);
                if (t >= total) break;
                next = (int)atomicAdd(fs.counter, 1u);  // its latency hides behind this tile's loads
                bool l1;
                int mt, nt;
                decode(t, l1, mt, nt);
                const GemmArgs& p = l1 ? p1 : p2;
                const CUtensorMap* tmA = l1 ? &tmA1 : &tmA2;
                const CUtensorMap* tmAs = l1 ? &tmA1s : &tmA2s;
                const CUtensorMap* tmB = l1 ? &tmB1 : &tmB2;
                const int e = p1.tile_expert ? p1.tile_expert[mt] : 0;
                const int row0 = p1.tile_row ? p1.tile_row[mt] : mt * BM;  // a multiple of 128
                if (!l1) {
                    // the L2 input of this row tile is complete once every L1 epilogue warp published it
                    if (!flag_wait_geq(fs.done + mt, done_target, tmo, abort_flag)) {
                        give_up();
                        break;
                    }
                    fence_proxy_async_global();
                }
                // A row tile with at most 96 used rows loads only the 32-row boxes holding
                // them (the rest of the A tile keeps stale bytes, whose accumulator rows no
                // epilogue stores); a fuller one loads the whole tile in one box.
                int used = BM;
                if (p1.seg_off) used = p1.seg_off[e] + p1.seg_cnt[e] - row0;
                else if (p1.counts) used = p1.counts[e] - (row0 - e * p1.rows_per_expert);
                else if (!p1.src) used = p1.m_valid - row0;
                const bool whole = used > BM - A_BOX_ROWS;
                const int a_boxes = whole ? 0 : (used <= A_BOX_ROWS ? 1 : (used + A_BOX_ROWS - 1) / A_BOX_ROWS);
                const uint32_t tx =
                    whole ? C::TX_BYTES : C::TX_BYTES - (uint32_t)(BM - a_boxes * A_BOX_ROWS) * BK_BYTES;
                bool ok = true;
                for (int ks = 0; ks < p.nks; ++ks) {
                    const uint32_t full = bar0 + 8 * stage, empty = bar0 + 8 * (STAGES + stage);
                    if (!mbar_wait(empty, phase ^ 1, tmo, abort_flag)) {
                        give_up();
                        ok = false;
                        break;
                    }
                    const uint32_t st = smem_u32(smem + stage * C::STAGE_BYTES);
                    mbar_arrive_expect_tx(full, tx);
                    if (whole)
                        tma_load_2d(st, tmA, full, ks * BK_BYTES, row0);
                    else
                        for (int b = 0; b < a_boxes; ++b)
                            tma_load_2d(st + b * (A_BOX_ROWS * BK_BYTES), tmAs, full, ks * BK_BYTES,
                                        row0 + b * A_BOX_ROWS);
                    tma_load_3d_hint(st + C::A_BYTES, tmB, full, ks * BK_BYTES, nt * BN, e,
                                     whole ? pol_reused : pol_once);
                    if constexpr (S > 0) {
                        bulk_load(st + C::A_BYTES + C::B_BYTES,
                                  p.sfa + ((int64_t)(row0 / BM) * p.nks + ks) * C::SFA_BYTES, C::SFA_BYTES, full);
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
                if (!ok) break;
            }
            // every load this thread issued lands before the CTA may exit
            for (int s = 0; s < STAGES; ++s)
                if (last_parity[s] >= 0) mbar_wait(bar0 + 8 * s, (uint32_t)last_parity[s], DRAIN_TIMEOUT_NS, never);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int k = 0;; ++k) {
                const int r = k % TRING;
                if (!mbar_wait(tile_full0 + 8 * r, (k / TRING) & 1, tmo, abort_flag)) {
                    give_up();
                    break;
                }
                const int t = tile_slot[r];
                mbar_arrive(tile_empty0 + 8 * r);
                if (t < 0) break;
                bool l1;
                int mt, nt;
                decode(t, l1, mt, nt);
                const int nks = l1 ? p1.nks : p2.nks;
                if (!mbar_wait(tempty_bar, acc_phase ^ 1, tmo, abort_flag)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                bool ok = true;
                for (int ks = 0; ks < nks; ++ks) {
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
                    if constexpr (SFW) {
                        // the scale-factor warps have written this stage's scale factors to tensor memory
                        if (!mbar_wait(sf_full0 + 8 * stage, phase, tmo, abort_flag)) {
                            give_up();
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    } else if constexpr (S > 0) {
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
                            mma_bf16(tmem_base, ad, bd, idesc_bf16(BN), accumulate);
                        else if constexpr (FMT == MOE_FMT_MXFP4)
                            mma_mxf4(tmem_base, ad, bd, idesc_mxf4(BN, 2u * (j & 1)), sfa_col + 4 * (j >> 1),
                                     sfb_col + 4 * NB * (j >> 1), accumulate);
                        else if constexpr (FMT == MOE_FMT_MXFP8)
                            mma_mxf8(tmem_base, ad, bd, idesc_mxf8(BN, j), sfa_col, sfb_col, accumulate);
                        else
                            mma_nvf4(tmem_base, ad, bd, idesc_nvf4(BN), sfa_col + 4 * j, sfb_col + 4 * NB * j,
                                     accumulate);
                    }
                    tc_commit(empty);
                    if (++stage == STAGES) {
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
            mbar_wait(drain_bar, 0, DRAIN_TIMEOUT_NS, never);
        }
    } else if (warp < 2 + EPI_WARPS) {
        const int q = warp % 4;           // the lane quarter of tensor memory this warp may read
        const int cg = (warp - 2) / 4;    // which quarter of the tile's columns it handles
        uint32_t acc_phase = 0;
        for (int k = 0;; ++k) {
            const int r = k % TRING;
            // warp-uniform: every lane leaves together (a lane left behind would block in __syncwarp)
            if (!__all_sync(0xffffffffu, mbar_wait(tile_full0 + 8 * r, (k / TRING) & 1, tmo, abort_flag))) {
                give_up();
                break;
            }
            const int t = tile_slot[r];
            __syncwarp();
            if (lane == 0) mbar_arrive(tile_empty0 + 8 * r);
            if (t < 0) break;
            bool l1;
            int mt, nt;
            decode(t, l1, mt, nt);
            if (!__all_sync(0xffffffffu, mbar_wait(tfull_bar, acc_phase, tmo, abort_flag))) {
                give_up();
                break;
            }
            tc_fence_after();
            const int e = p1.tile_expert ? p1.tile_expert[mt] : 0;
            const int row = (p1.tile_row ? p1.tile_row[mt] : mt * BM) + q * 32 + lane;
            const uint32_t tacc = tmem_base + ((uint32_t)(q * 32) << 16);
            // hand the accumulator back as soon as it sits in registers
            auto release = [&]() {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar);
            };
            if (l1) {
                epilogue_l1<FMT, BN>(p1, tacc, row, nt, e, cg, release);
                // publish this warp's rows of the L2 input to the producers of L2 tiles
                __threadfence();
                fence_proxy_async_global();
                __syncwarp();
                if (lane == 0) red_release_gpu_add(fs.done + mt, 1u);
            } else {
                epilogue_l2<FMT, BN>(p2, tacc, row, nt, e, cg, release);
            }
            acc_phase ^= 1;
        }
    } else if constexpr (SFW) {
        // Scale-factor warps, one per lane quarter of tensor memory (warps 18..21: quarters
        // 2, 3, 0, 1). For each stage, once it has landed, a warp stores the stage's scale
        // atoms into its own quarter with tcgen05.st, in the layout a 32x128b.warpx4 copy of
        // each atom gives: lane i, columns 4 a .. 4 a + 3 <- bytes 16 i .. 16 i + 15 of the
        // atom copied to column 4 a. Then the MMA thread issues only MMAs. A stage's columns
        // are written again only after its next fill has landed, which follows the commit
        // of the MMAs that read them.
        const int q = warp % 4;
        const uint32_t quarter = tmem_base + ((uint32_t)(q * 32) << 16);
        int stage = 0;
        uint32_t phase = 0;
        for (int k = 0;; ++k) {
            const int r = k % TRING;
            if (!__all_sync(0xffffffffu, mbar_wait(tile_full0 + 8 * r, (k / TRING) & 1, tmo, abort_flag))) {
                give_up();
                break;
            }
            const int t = tile_slot[r];
            __syncwarp();
            if (lane == 0) mbar_arrive(tile_empty0 + 8 * r);
            if (t < 0) break;
            const int nks = t < total1 ? p1.nks : p2.nks;
            bool ok = true;
            for (int ks = 0; ks < nks; ++ks) {
                if (!__all_sync(0xffffffffu, mbar_wait(bar0 + 8 * stage, phase, tmo, abort_flag))) {
                    give_up();
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t* sf = smem + stage * C::STAGE_BYTES + C::A_BYTES + C::B_BYTES;
                const uint32_t col = quarter + C::ACC_COLS + stage * C::SF_COLS;
#pragma unroll
                for (int a = 0; a < S; ++a)
                    tmem_st4(col + 4 * a, *reinterpret_cast<const uint4*>(sf + a * ATOM_BYTES + 16 * lane));
                // smem holds the weight atoms as [block][s]; tensor memory wants [s][block]
#pragma unroll
                for (int a = 0; a < S; ++a)
#pragma unroll
                    for (int nb = 0; nb < NB; ++nb)
                        tmem_st4(col + 4 * S + 4 * (a * NB + nb),
                                 *reinterpret_cast<const uint4*>(sf + C::SFA_BYTES + (nb * S + a) * ATOM_BYTES +
                                                                 16 * lane));
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(sf_full0 + 8 * stage);
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
    // the successor's own wait covers this kernel only: this grid completes after the
    // previous one
    if (fs.independent) grid_dep_wait();
}

// ------------------------------------------------------------------ host side
template <int FMT>
static cudaError_t fused_attr() {
    return cudaFuncSetAttribute(fused_mlp_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                FusedCfg<FMT>::SMEM);
}

cudaError_t fused_prepare(int fmt) {
    switch (fmt) {
        case MOE_FMT_BF16: return fused_attr<MOE_FMT_BF16>();
        case MOE_FMT_MXFP8: return fused_attr<MOE_FMT_MXFP8>();
        case MOE_FMT_MXFP4: return fused_attr<MOE_FMT_MXFP4>();
        default: return fused_attr<MOE_FMT_NVFP4>();
    }
}

template <int FMT>
static cudaError_t fused_t(const CUtensorMap& a1, const CUtensorMap& b1, const CUtensorMap& a2,
                           const CUtensorMap& b2, const CUtensorMap& a1s, const CUtensorMap& a2s, const GemmArgs& p1,
                           const GemmArgs& p2, const FusedSched& fs, int grid, cudaStream_t st, bool pdl) {
    LaunchAttrs at(pdl);
    cudaLaunchConfig_t cfg = at.config(dim3(grid), dim3(FusedCfg<FMT>::THREADS), FusedCfg<FMT>::SMEM, st);
    return cudaLaunchKernelEx(&cfg, fused_mlp_kernel<FMT>, a1, b1, a2, b2, a1s, a2s, p1, p2, fs);
}

cudaError_t launch_fused_mlp(int fmt, const CUtensorMap& a1, const CUtensorMap& b1, const CUtensorMap& a2,
                             const CUtensorMap& b2, const CUtensorMap& a1s, const CUtensorMap& a2s,
                             const GemmArgs& p1, const GemmArgs& p2, const FusedSched& fs, int grid, cudaStream_t st,
                             bool pdl) {
    switch (fmt) {
        case MOE_FMT_BF16: return fused_t<MOE_FMT_BF16>(a1, b1, a2, b2, a1s, a2s, p1, p2, fs, grid, st, pdl);
        case MOE_FMT_MXFP8: return fused_t<MOE_FMT_MXFP8>(a1, b1, a2, b2, a1s, a2s, p1, p2, fs, grid, st, pdl);
        case MOE_FMT_MXFP4: return fused_t<MOE_FMT_MXFP4>(a1, b1, a2, b2, a1s, a2s, p1, p2, fs, grid, st, pdl);
        default: return fused_t<MOE_FMT_NVFP4>(a1, b1, a2, b2, a1s, a2s, p1, p2, fs, grid, st, pdl);
    }
}

}  // namespace moe
