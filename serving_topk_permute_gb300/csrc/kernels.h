// kernels.h -- internal host-side launchers of the MoE kernels (not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// Launch attributes: programmatic stream serialisation (pdl) and an optional cluster
// size. The attribute array must outlive the launch call only.
struct LaunchAttrs {
    cudaLaunchAttribute a[2];
    int n = 0;
    LaunchAttrs(bool pdl, int cluster = 1) {
        if (pdl) {
            a[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            a[n].val.programmaticStreamSerializationAllowed = 1;
            ++n;
        }
        if (cluster > 1) {
            a[n].id = cudaLaunchAttributeClusterDimension;
            a[n].val.clusterDim.x = (unsigned)cluster;
            a[n].val.clusterDim.y = 1;
            a[n].val.clusterDim.z = 1;
            ++n;
        }
    }
    cudaLaunchConfig_t config(dim3 grid, dim3 block, size_t smem, cudaStream_t st) {
        cudaLaunchConfig_t c = {};
        c.gridDim = grid;
        c.blockDim = block;
        c.dynamicSmemBytes = smem;
        c.stream = st;
        c.attrs = a;
        c.numAttrs = (unsigned)n;
        return c;
    }
};

// ------------------------------------------------------------------ routing
// Histogram, BLOCK_M (bm)-padded offsets, stable scatter (one CTA). Writes cnt[E],
// off[E+1], src[r] = -1 for the padding rows only (the routed rows are src[inv[s]] = s,
// written by the dispatch kernel), inv[T*k] (-1 masked), tile_expert[M_pad/bm],
// meta[0] = M_pad, meta[1] = M_pad / bm.
size_t route_smem_bytes(int E);
cudaError_t route_prepare(int E);   // sets the dynamic shared memory attribute (E <= 512)
// zero[0..n_zero): words the routing kernel also zeroes (the GEMM schedule counters).
// With wbase ([ROUTE_WARPS][E] ints), the kernel writes each slot chunk's first row in
// each expert there and leaves inv (and the routed rows of src) to the dispatch kernel;
// without it, it writes inv itself.
cudaError_t launch_route(const int32_t* ids, int T, int k, int E, int bm, int* cnt, int* off, int* src, int* inv,
                         int* tile_expert, int* meta, int* err, cudaStream_t st, bool pdl = false,
                         uint32_t* zero = nullptr, int n_zero = 0, int* wbase = nullptr);

// Batched (masked) layout: the row tiles holding used rows (counts[e] of expert e's
// M-row slab), in expert order: tile_expert[], tile_row[] (first row), meta[1] = number
// of tiles; row_prefix[E+1] = used rows of the experts before e. Also zeroes err and
// zero[0..n_zero). One CTA; E <= 1024.
cudaError_t launch_batched_plan(const int32_t* counts, int E, int M, int* tile_expert, int* tile_row,
                                int* row_prefix, int* meta, int* err, uint32_t* zero, int n_zero, cudaStream_t st,
                                bool pdl = false);

// ------------------------------------------------------------------ dispatch quantisation
struct DispatchArgs {
    const uint16_t* x;   // bf16 bits [T, H]
    int T, H, k;
    const int32_t* ids;  // [T*k] expert of each slot
    int E;
    const int* wbase;    // [ROUTE_WARPS][E] first row of each slot chunk in each expert (routing)
    int* inv;            // [T*k] written here: permuted row of each slot (-1 = masked)
    int* src;            // [M_pad] written here for the routed rows: src[inv[s]] = s
    int fmt;             // routed format
    uint8_t* xq;         // [M_pad_max, H/vpe] permuted rows
    uint8_t* xsf;        // scale atoms
    float* x_scale;      // [T] NVFP4 per-token scale
    int shared_fmt;      // -1: no shared copy
    uint8_t* sxq;        // [T_pad, H/vpe] identity rows
    uint8_t* sxsf;
    // batched layout (when batch_counts is set): T = E * batch_M rows, row e * M + m used
    // when m < batch_counts[e], quantised into the same row; no ranks, no shared copy.
    // batch_prefix[E+1] (from the planning kernel): used rows of the experts before e.
    const int* batch_counts;
    const int* batch_prefix;
    int batch_M;
};
cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t st, bool pdl = false);

// ------------------------------------------------------------------ grouped GEMM
struct GemmArgs {
    const uint8_t* sfa;        // activation scale atoms [row tiles][nks][S][512]
    const uint8_t* sfb;        // weight scale atoms [E][nks][sf_blocks][S][512]
    int nks;                   // 128-byte K stages
    int n_tiles;               // BN-column tiles
    int sf_blocks;             // 128-row blocks of the weight scale layout (wt_sf_blocks(N))
    int N;                     // output columns (kernel-layout weight rows)
    const int* m_tiles_dev;    // number of 128-row tiles on the device (or null)
    int m_tiles_host;          // used when m_tiles_dev is null
    const int* tile_expert;    // expert of each row tile (null: expert 0)
    const int* tile_row;       // first row of each row tile (null: tile * 128)
    const int* src;            // flat slot of each row, -1 = padding (null: see counts, else rows < m_valid)
    int m_valid;
    const int* seg_off;        // routed layout: first row [E] and row count [E] of each expert's segment
    const int* seg_cnt;        //   (null: the row tile's used rows follow from counts or m_valid)
    const int* counts;         // batched layout: row r is used when r % rows_per_expert < counts[r / rows_per_expert]
    int rows_per_expert;
    int top_k;
    const float* x_scale;      // NVFP4 L1: per-token dispatch scale [T]
    const float* gscale;       // NVFP4: per-expert global weight scale [E]
    const float* a2;           // NVFP4: device scalar, the L2 input scale
    // L1 epilogue output (the L2 input)
    uint8_t* hq;
    uint8_t* hsf;
    int I;
    int h_nks;
    float* h_debug;
    float act_alpha, act_beta, act_clamp;
    int act_has_clamp;
    // L2 epilogue output
    __nv_bfloat16* y;
    int ldy;
    int* err;
    unsigned long long timeout_ns;
};
cudaError_t gemm_prepare(int fmt);   // sets the dynamic shared memory attribute of every variant

// Both GEMMs in one persistent kernel (256-wide tiles, single CTAs). counter: the
// next tile to take; done[m_tiles]: published L1 epilogue warps per row tile. Both
// must be zero at launch (the routing kernel zeroes them). a1/a2 load A tiles as one
// 128-row box, a1s/a2s (same tensors) as A_BOX_ROWS-row boxes for mostly empty tiles.
struct FusedSched {
    uint32_t* counter;
    uint32_t* done;
    // 1: the kernel reads nothing the kernel launched just before it writes (the shared
    // expert after the routed GEMMs). It then takes its tiles as soon as it is resident
    // and waits for that kernel only before it exits, so its successor still finds both
    // complete.
    int independent;
};
cudaError_t fused_prepare(int fmt);
cudaError_t launch_fused_mlp(int fmt, const CUtensorMap& a1, const CUtensorMap& b1, const CUtensorMap& a2,
                             const CUtensorMap& b2, const CUtensorMap& a1s, const CUtensorMap& a2s,
                             const GemmArgs& p1, const GemmArgs& p2, const FusedSched& fs, int grid, cudaStream_t st,
                             bool pdl = false);
// CTA-pair variant: 256 x 256 tiles over 256-row segments; the B map's box is 128 rows
cudaError_t gemm2_prepare(int fmt);
// tmSFA / tmSFB: the scale atoms as 2-D uint32 tensors [atoms][128] with boxes of
// S (activation) and S * 2 (weight) atoms; unused for BF16
cudaError_t launch_gemm2(int fmt, bool l1, const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmSFA,
                         const CUtensorMap& tmSFB, const GemmArgs& a, int grid, cudaStream_t st, bool pdl = false);
// bn: 128 or 256 (the tile width; the B tensor map's box must be bn rows)
cudaError_t launch_gemm(int fmt, bool l1, int bn, const CUtensorMap& tmA, const CUtensorMap& tmB, const GemmArgs& a,
                        int grid, cudaStream_t st, bool pdl = false);

// ------------------------------------------------------------------ combine
struct CombineArgs {
    const __nv_bfloat16* y;    // [M_pad_max, H] per-row L2 output
    const int* inv;            // [T*k]
    const float* w;            // [T*k]
    int T, k, H;
    const __nv_bfloat16* ys;   // [T, H] shared expert output or null
    const float* gamma;        // [H] or null
    float eps;
    __nv_bfloat16* out;        // [T, H]
};
cudaError_t combine_prepare();   // allows the norm's [H] fp32 shared-memory row (H <= 16384)
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t st, bool pdl = false);

// ------------------------------------------------------------------ weight transform
cudaError_t launch_interleave_rows(const uint8_t* src, uint8_t* dst, int E, int I, int64_t row_bytes,
                                   cudaStream_t st);
// scale atoms from row-major [E, N, K/g] u8 scales; interleave: apply the w13 row interleave
cudaError_t launch_pack_weight_sf(const uint8_t* src, uint8_t* dst, int fmt, int E, int N, int K, bool interleave,
                                  int I, cudaStream_t st);

}  // namespace moe
