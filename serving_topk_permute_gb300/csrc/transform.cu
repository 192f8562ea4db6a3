// transform.cu -- one-time repack of checkpoint weights into the kernel layout
// (vllm.models.muse_spark.nvidia.mega_moe, finalize_weights ->
// transform_weights_for_mega_moe; vllm.model_executor.layers.fused_moe.
// deep_gemm_mega_moe, DeepGemmMegaMoEExperts._kernel_layout_shard / _pack_scale).
//
//   rows   w13 rows are interleaved per 128-row block so that every 128-row
//          block holds 64 gate rows and the 64 matching up rows: kernel row
//          128b + 64h + r <- checkpoint row h*I + 64b + r (the pages interleave
//          by 8 rows); a 128- or 256-wide MMA N tile then holds whole gate/up
//          pairs
//   scales row-major [N, K/g] bytes -> 512-byte atoms for the tensor-memory copy:
//          128 rows x 4 scale blocks, row 32j + i / scale b at byte 16i + 4j + b
//          (the pages' UTCCP permutation: row 128b + 32j + i -> 128b + 4i + j),
//          atoms ordered [E][K stage][N blocks][S] so that one K stage of any
//          128- or 256-row tile is a single contiguous bulk copy. Rows past N are zero.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// one CTA per (expert, kernel row), 16 bytes per thread per step
__global__ void interleave_rows_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int I,
                                       int64_t row_bytes) {
    const int64_t e = blockIdx.y;
    const int n = blockIdx.x;  // kernel row in [0, 2I)
    const int64_t src_row = w13_src_row(n, I);
    const uint4* s = reinterpret_cast<const uint4*>(src + (e * 2 * I + src_row) * row_bytes);
    uint4* d = reinterpret_cast<uint4*>(dst + (e * 2 * I + n) * row_bytes);
    for (int64_t i = threadIdx.x; i < row_bytes / 16; i += blockDim.x) d[i] = s[i];
}

cudaError_t launch_interleave_rows(const uint8_t* src, uint8_t* dst, int E, int I, int64_t row_bytes,
                                   cudaStream_t st) {
    if (E == 0) return cudaSuccess;
    dim3 grid(2 * I, E);
    interleave_rows_kernel<<<grid, 128, 0, st>>>(src, dst, I, row_bytes);
    return cudaGetLastError();
}

// one thread per destination byte
__global__ void pack_weight_sf_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t total, int S,
                                      int64_t nks, int64_t n_blocks, int N, int nkb, int interleave, int I) {
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    int64_t q = idx;
    const int in_atom = (int)(q % ATOM_BYTES);
    q /= ATOM_BYTES;
    const int s = (int)(q % S);
    q /= S;
    const int64_t nb = q % n_blocks;
    q /= n_blocks;
    const int64_t ks = q % nks;
    const int64_t e = q / nks;
    const int i = in_atom / 16, j = (in_atom % 16) / 4, b = in_atom % 4;
    const int64_t n = nb * NBLK + j * 32 + i;          // kernel-layout row
    const int64_t kb = ks * 4 * S + s * 4 + b;          // scale block along K
    uint8_t v = 0;
    if (n < N && kb < nkb) {
        const int64_t row = interleave ? w13_src_row(n, I) : n;
        v = src[(e * N + row) * nkb + kb];
    }
    dst[idx] = v;
}

cudaError_t launch_pack_weight_sf(const uint8_t* src, uint8_t* dst, int fmt, int E, int N, int K, bool interleave,
                                  int I, cudaStream_t st) {
    const int S = fmt_sf_atoms(fmt);
    if (S == 0 || E == 0) return cudaSuccess;
    const int64_t nks = fmt_k_stages(fmt, K);
    const int64_t n_blocks = wt_sf_blocks(N);
    const int64_t total = (int64_t)E * nks * n_blocks * S * ATOM_BYTES;
    const int nkb = K / fmt_sf_block(fmt);
    const int threads = 256;
    pack_weight_sf_kernel<<<(unsigned)ceil_div(total, threads), threads, 0, st>>>(src, dst, total, S, nks, n_blocks, N,
                                                                                 nkb, interleave ? 1 : 0, I);
    return cudaGetLastError();
}

}  // namespace moe
