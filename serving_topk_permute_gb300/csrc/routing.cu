// routing.cu -- per-expert histogram, BLOCK_M-padded segment offsets and the stable
// scatter of routed slots into them (vllm.model_executor.layers.fused_moe,
// DeepGemmExperts.workspace_shapes: compute_aligned_M, M_sum % block_m == 0;
// DeepGemmExperts.apply: deepgemm_moe_permute -> expert ids and inv_perm).
//
// Segments are padded to BLOCK_M = bm rows (128, or 256 for the CTA-pair GEMM).
// One CTA of 1024 threads (32 warps). Warp w owns a contiguous chunk of the
// flat slots s = t*k + j.
//   pass 1  each warp counts its chunk per expert into its own shared row
//   scan    per expert, one warp by shuffles: exclusive prefix over the 32 warps'
//           counts (a warp's base inside the expert) and the total; padded
//           sizes; a block-wide scan gives the segment offsets; the padding rows
//           are marked -1
//   pass 2  each warp walks its chunk in ascending order, 32 slots at a time;
//           __match_any_sync groups lanes with the same expert, the rank inside
//           the group plus the warp's running count gives the row, stored as
//           inv_perm[slot] (coalesced). Rows inside a segment are therefore
//           ordered by ascending slot: a stable scatter. The inverse, src[row],
//           is written by the dispatch kernel, one token's slots per CTA: as
//           scattered 4-byte stores from this one CTA it took most of the time.
// Integer-only and deterministic. Ids outside [-1, E) set MOE_ERR_BAD_EXPERT_ID
// and are treated as masked.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int ROUTE_THREADS = 32 * ROUTE_WARPS;
constexpr int RB = 8;  // 32-slot groups whose ids are loaded together

__global__ void __launch_bounds__(ROUTE_THREADS, 1)
    route_kernel(const int32_t* __restrict__ ids, int T, int k, int E, int bm, int* __restrict__ cnt,
                 int* __restrict__ off, int* __restrict__ src, int* __restrict__ inv, int* __restrict__ tile_expert,
                 int* __restrict__ meta, int* err, uint32_t* __restrict__ zero, int n_zero,
                 int* __restrict__ wbase, bool scatter) {
    extern __shared__ int sm[];
    const int WS = E | 1;                    // odd row stride: a warp reading one expert's 32 rows hits 32 banks
    int* wcnt = sm;                          // [32][WS]: per-warp counts, then per-warp running bases
    int* s_off = sm + ROUTE_WARPS * WS;      // [E+1]
    int* s_cnt = s_off + (E + 1);            // [E]
    int* s_wsum = s_cnt + E;                 // [32] scan scratch
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int R = T * k;
    const int chunk = route_chunk(R);
    const int beg = min(warp * chunk, R), end = min(beg + chunk, R);

    for (int i = tid; i < ROUTE_WARPS * WS; i += ROUTE_THREADS) wcnt[i] = 0;
    grid_dep_wait();  // the previous kernel (which may still read src / inv) has finished
    grid_dep_launch();
    if (tid == 0 && err) *err = 0;  // the status word reflects this forward only
    for (int i = tid; i < n_zero; i += ROUTE_THREADS) zero[i] = 0u;
    __syncthreads();

    // pass 1: per-warp histograms (ids loaded RB groups of 32 at a time: independent loads in
    // flight). A warp whose chunk is one batch keeps its ids in registers for pass 2.
    const bool one_batch = end - beg <= 32 * RB;
    int kept[RB];
    for (int s0 = beg; s0 < end; s0 += 32 * RB) {
        int ev[RB];
#pragma unroll
        for (int u = 0; u < RB; ++u) {
            const int s = s0 + 32 * u + lane;
            ev[u] = s < end ? ids[s] : -1;
            kept[u] = ev[u];
        }
#pragma unroll
        for (int u = 0; u < RB; ++u) {
            if (s0 + 32 * u >= end) break;  // warp-uniform
            const int e = ev[u];
            if (e >= 0 && e < E)
                atomicAdd(&wcnt[warp * WS + e], 1);
            else if (e != -1)
                set_error(err, MOE_ERR_BAD_EXPERT_ID);
        }
    }
    __syncthreads();

    // per expert (one warp each): exclusive prefix of its 32 per-warp counts by shuffles,
    // the total, and the padded size
    for (int e = warp; e < E; e += ROUTE_WARPS) {
        const int c = wcnt[lane * WS + e];
        int x = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        wcnt[lane * WS + e] = x - c;
        if (lane == 31) {
            s_cnt[e] = x;
            cnt[e] = x;
        }
    }
    __syncthreads();

    // block-wide exclusive scan of the padded sizes (E <= 1024: one value per thread)
    {
        const int v = tid < E ? (int)align_up(s_cnt[tid], bm) : 0;
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) s_wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = s_wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            s_wsum[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int incl = x + (warp > 0 ? s_wsum[warp - 1] : 0);
        if (tid < E) s_off[tid] = incl - v;
        if (tid == E - 1) s_off[E] = incl;
    }
    __syncthreads();
    for (int e = tid; e <= E; e += ROUTE_THREADS) off[e] = s_off[e];
    // each chunk's first row in each expert (its base); the dispatch kernel adds a slot's
    // rank inside the chunk
    if (wbase)
        for (int i = tid; i < ROUTE_WARPS * E; i += ROUTE_THREADS)
            wbase[i] = s_off[i % E] + wcnt[(i / E) * WS + i % E];
    // the padding rows of each segment (one warp per expert); the scatter below writes the rest
    for (int e = warp; e < E; e += ROUTE_WARPS)
        for (int r = s_off[e] + s_cnt[e] + lane; r < s_off[e + 1]; r += 32) src[r] = -1;

    // pass 2: stable scatter, in ascending slot order (ids again loaded RB groups at a time,
    // unless still in registers)
    const unsigned lt = (1u << lane) - 1u;
    for (int s0 = beg; scatter && s0 < end; s0 += 32 * RB) {
        int ev[RB];
#pragma unroll
        for (int u = 0; u < RB; ++u) {
            const int s = s0 + 32 * u + lane;
            ev[u] = one_batch ? kept[u] : (s < end ? ids[s] : -1);
        }
#pragma unroll
        for (int u = 0; u < RB; ++u) {
            if (s0 + 32 * u >= end) break;  // warp-uniform
            const int s = s0 + 32 * u + lane;
            const int e = ev[u];
            const bool routed = s < end && e >= 0 && e < E;
            const int key = routed ? e : E + lane;  // unrouted lanes never group
            const unsigned peers = __match_any_sync(0xffffffffu, key);
            if (s < end) inv[s] = routed ? s_off[e] + wcnt[warp * WS + e] + __popc(peers & lt) : -1;
            __syncwarp();
            if (routed && lane == __ffs(peers) - 1) wcnt[warp * WS + e] += __popc(peers);
            __syncwarp();
        }
    }

    // the row-tile -> expert map
    for (int e = tid; e < E; e += ROUTE_THREADS)
        for (int mt = s_off[e] / bm; mt < s_off[e + 1] / bm; ++mt) tile_expert[mt] = e;
    if (tid == 0) {
        meta[0] = s_off[E];
        meta[1] = s_off[E] / bm;
    }
}

size_t route_smem_bytes(int E) { return sizeof(int) * ((size_t)ROUTE_WARPS * (E | 1) + (E + 1) + E + 32); }

cudaError_t route_prepare(int E) {
    return cudaFuncSetAttribute(route_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)route_smem_bytes(E));
}

cudaError_t launch_route(const int32_t* ids, int T, int k, int E, int bm, int* cnt, int* off, int* src, int* inv,
                         int* tile_expert, int* meta, int* err, cudaStream_t st, bool pdl, uint32_t* zero,
                         int n_zero, int* wbase) {
    LaunchAttrs at(pdl);
    cudaLaunchConfig_t cfg = at.config(dim3(1), dim3(ROUTE_THREADS), route_smem_bytes(E), st);
    return cudaLaunchKernelEx(&cfg, route_kernel, ids, T, k, E, bm, cnt, off, src, inv, tile_expert, meta, err, zero,
                              n_zero, wbase, wbase == nullptr);
}

}  // namespace moe

namespace moe {

// Batched (masked) layout (vllm.model_executor.layers.fused_moe, BatchedDeepGemmExperts:
// m-grouped GEMMs over [E, max_num_tokens, K] with expert_num_tokens[E]): the row tiles
// that hold used rows, in expert order. Expert e's slab is rows [e M, e M + M); its first
// counts[e] rows are used, so it contributes ceil(counts[e] / 128) row tiles. One CTA.
__global__ void __launch_bounds__(ROUTE_THREADS, 1)
    batched_plan_kernel(const int32_t* __restrict__ counts, int E, int M, int* __restrict__ tile_expert,
                        int* __restrict__ tile_row, int* __restrict__ row_prefix, int* __restrict__ meta, int* err,
                        uint32_t* __restrict__ zero, int n_zero) {
    __shared__ int s_wsum[ROUTE_WARPS];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    grid_dep_wait();  // the previous kernel (which may still read the tile lists) has finished
    grid_dep_launch();
    if (tid == 0 && err) *err = 0;
    for (int i = tid; i < n_zero; i += ROUTE_THREADS) zero[i] = 0u;
    __syncthreads();
    int n = 0, c = 0;
    if (tid < E) {
        c = counts[tid];
        if (c < 0 || c > M) {
            set_error(err, MOE_ERR_CAPACITY);
            c = c < 0 ? 0 : M;
        }
        n = (c + BM - 1) / BM;
    }
    // block-wide exclusive scan of the tile counts (E <= 1024: one value per thread)
    int x = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = s_wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        s_wsum[lane] = w;
    }
    __syncthreads();
    const int incl = x + (warp > 0 ? s_wsum[warp - 1] : 0);
    for (int j = 0; j < n; ++j) {
        tile_expert[incl - n + j] = tid;
        tile_row[incl - n + j] = tid * M + j * BM;
    }
    if (tid == ROUTE_THREADS - 1) {
        meta[0] = incl * BM;
        meta[1] = incl;
    }
    // the same scan over the used rows: row_prefix[e] = used rows of experts before e, so
    // the dispatch kernel can spread the used rows evenly over its CTAs
    __syncthreads();
    x = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = s_wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        s_wsum[lane] = w;
    }
    __syncthreads();
    const int rincl = x + (warp > 0 ? s_wsum[warp - 1] : 0);
    if (tid < E) row_prefix[tid] = rincl - c;
    if (tid == E - 1) row_prefix[E] = rincl;
}

cudaError_t launch_batched_plan(const int32_t* counts, int E, int M, int* tile_expert, int* tile_row,
                                int* row_prefix, int* meta, int* err, uint32_t* zero, int n_zero, cudaStream_t st,
                                bool pdl) {
    LaunchAttrs at(pdl);
    cudaLaunchConfig_t cfg = at.config(dim3(1), dim3(ROUTE_THREADS), 0, st);
    return cudaLaunchKernelEx(&cfg, batched_plan_kernel, counts, E, M, tile_expert, tile_row, row_prefix, meta, err,
                              zero, n_zero);
}

}  // namespace moe
