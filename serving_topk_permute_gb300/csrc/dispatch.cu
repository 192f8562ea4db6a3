// dispatch.cu -- dispatch-side activation quantisation fused with the permute
// (vllm.model_executor.layers.fused_moe.deep_gemm_mega_moe, module docstring and
// DeepGemmMegaMoEExperts.forward: prepare_megamoe_inputs quantises hidden once
// per token; vllm.model_executor.layers.fused_moe, DeepGemmExperts.apply:
// deepgemm_moe_permute writes a1q_perm).
//
// One CTA per token: 128 threads for H <= 4096 and T >= 1024, else 256. Each thread owns 8-element
// chunks c = tid + NT i of the row (NT threads; at most 4 of them for H <= 8192, 8
// above), loaded as one 128-bit bf16x8 vector each, kept in registers. Per format:
//   BF16   the 16-byte chunk is copied as is
//   MXFP8  a 32-element block is 4 neighbouring threads: block amax by two xor
//          shuffles, e = smallest integer with amax <= 448 * 2^e, codes
//          E4M3(x * 2^-e) (RNE, saturating), scale byte e + 127
//   NVFP4  token amax by a block reduction, token scale gs = amax / 2688 (fp32),
//          a 16-element block is 2 neighbouring threads: block scale
//          sb = E4M3(amax_b / (gs * 6)), eff = value(sb) * gs, codes E2M1(x / eff)
//          packed two per byte (element 2i in the low nibble), all in fp32 RN
// The codes are written to each of the token's k permuted rows (inv_perm), and
// the scale bytes to the matching position of the 128-row scale atoms the MMA
// reads. With a shared expert, the token is also quantised to the shared format
// into row t of a separate (unpermuted) buffer.
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int DISPATCH_THREADS = 256;
constexpr int DISPATCH_MAX_CHUNKS = 8;   // H <= 8 * 256 * 8 = 16384
// Rows of H <= 8192 use a variant holding 4 chunks per thread, which fits in 48
// registers, so that 5 CTAs (tokens) are resident per SM instead of 3.
constexpr int DISPATCH_SMALL_CHUNKS = 4;
constexpr int DISPATCH_SMALL_MIN_CTAS = 5;
// Rows of H <= 4096 in batches too large to be resident at once use CTAs of 128 threads
// (4 chunks each), twice as many tokens in flight per SM. Smaller batches keep 256 threads:
// there every CTA is resident anyway, and a narrower CTA only lengthens each thread's work.
constexpr int DISPATCH_NARROW_THREADS = 128;
constexpr int DISPATCH_NARROW_MIN_CTAS = 10;
constexpr int DISPATCH_NARROW_MIN_TOKENS = 1024;

__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

// 2^n exactly, for -149 <= n <= 127 (fp32 subnormals below 2^-126). x * pow2f(n) is then the
// correctly rounded x * 2^n, the value ldexpf(x, n) returns, at the cost of one multiply
// (this library builds with IEEE subnormals: no flush to zero).
__device__ __forceinline__ float pow2f(int n) {
    return n >= -126 ? __int_as_float((n + 127) << 23) : __int_as_float(1 << (n + 149));
}

// Row r's scale byte of block kb in the activation scale atoms (act_sf_offset) is
// sf_row_base(r) + (kb / 4) * 512 + kb % 4: each atom holds 4 blocks of 128 rows, and the
// atoms of a row tile follow one another in K order.
__device__ __forceinline__ int64_t sf_row_base(int64_t r, int S, int64_t nks) {
    return (r / BM) * nks * S * ATOM_BYTES + (r % 32) * 16 + ((r % BM) / 32) * 4;
}
__device__ __forceinline__ int64_t sf_byte(int64_t base, int kb) { return base + (int64_t)(kb >> 2) * ATOM_BYTES + (kb & 3); }

// MXFP8 codes of one 8-element chunk (block exponent ex), as 8 bytes
__device__ __forceinline__ uint2 mxfp8_chunk(const float (&f)[8], int ex) {
    const float sc = pow2f(-ex);  // ex in [-127, 127]
    uint32_t w[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t lo = cvt_e4m3x2(f[4 * i] * sc, f[4 * i + 1] * sc);
        const uint32_t hi = cvt_e4m3x2(f[4 * i + 2] * sc, f[4 * i + 3] * sc);
        w[i] = lo | (hi << 16);
    }
    return make_uint2(w[0], w[1]);
}

// block exponent of the 32-element block held by 4 neighbouring lanes
__device__ __forceinline__ int mxfp8_block_exponent(const float (&f)[8]) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    return ue8m0_exponent(amax);
}

// One token (routed layout: written to its k permuted rows) or one row of the batched
// layout (batched: written to the same row).
template <int MAXC, int NT>
__device__ __forceinline__ void dispatch_one(const DispatchArgs& a, const int t, const bool batched) {
    const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
    const int nchunks = a.H / 8;
    __shared__ int s_rows[32];
    __shared__ int64_t s_sfb[32];  // each row's scale-byte base in the atoms (sf_row_base)
    __shared__ int s_rank[32];  // rank of slot j among the equal ids before it in its routing chunk
    __shared__ int s_exp[32];
    __shared__ float s_amax[NT / 32];

    // The token's row and its own scale do not depend on routing. The hidden states are
    // complete before this kernel starts (routing, the kernel before it, lets it start only
    // after its own wait for its predecessor), so they are read while routing still runs.
    // load the token's row into registers
    uint4 v[MAXC];
    const uint4* xrow = reinterpret_cast<const uint4*>(a.x + (int64_t)t * a.H);
#pragma unroll
    for (int i = 0; i < MAXC; ++i) {
        const int c = tid + i * NT;
        v[i] = c < nchunks ? __ldcg(xrow + c) : make_uint4(0, 0, 0, 0);  // from L2: no stale L1 line
    }

    // Each slot's row is its routing chunk's first row in the expert (written by the
    // routing kernel) plus the number of equal ids before it in the chunk: a stable
    // scatter, counted here from the ids alone. The CTA scans the chunk's ids before this
    // token once (128-bit loads, 8 ids per thread per round), counting the token's k
    // experts, then adds the equal slots of the token itself that come first. (When k
    // does not divide 32 a token's slots may straddle two chunks; a slot in the second
    // chunk counts only the token's slots from that chunk's start.)
    const int R = a.T * a.k, chunk = route_chunk(R);
    const int s0 = t * a.k, c0 = s0 / chunk * chunk;
    if (!batched) {
    if (tid < a.k) {
        s_exp[tid] = __ldcg(a.ids + s0 + tid);
        s_rank[tid] = 0;
    }
    __syncthreads();
    for (int base = c0; base < s0; base += 8 * NT) {
        int v[8];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const int i0 = base + 4 * tid + 4 * NT * m;
            if (i0 + 3 < s0) {
                const int4 q = __ldcg(reinterpret_cast<const int4*>(a.ids + i0));
                v[4 * m] = q.x, v[4 * m + 1] = q.y, v[4 * m + 2] = q.z, v[4 * m + 3] = q.w;
            } else {
#pragma unroll
                for (int u = 0; u < 4; ++u) v[4 * m + u] = i0 + u < s0 ? __ldcg(a.ids + i0 + u) : INT_MIN;
            }
        }
        for (int j = 0; j < a.k; ++j) {
            const int e = s_exp[j];
            int n = 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) n += v[u] == e;
            n = __reduce_add_sync(0xffffffffu, n);
            if (lane == 0 && n) atomicAdd(&s_rank[j], n);
        }
    }
    __syncthreads();
    if (tid < a.k) {
        const int e = s_exp[tid], my_chunk = (s0 + tid) / chunk;
        int n = my_chunk == s0 / chunk ? s_rank[tid] : 0;
        for (int j = 0; j < tid; ++j) n += s_exp[j] == e && (s0 + j) / chunk == my_chunk;
        s_rank[tid] = n;  // only this thread reads it back (after the next barrier)
    }
    }  // !batched

    // NVFP4: the token's own scale
    float gs = 1.0f;
    if (a.fmt == MOE_FMT_NVFP4) {
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < MAXC; ++i) {
            float f[8];
            bf16x8_to_f32(v[i], f);
#pragma unroll
            for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        if (lane == 0) s_amax[warp] = amax;
        __syncthreads();
        amax = s_amax[0];
#pragma unroll
        for (int w = 1; w < NT / 32; ++w) amax = fmaxf(amax, s_amax[w]);
        gs = amax > 0.0f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
    }
    grid_dep_wait();  // routing has written the chunk bases (and the previous forward is done with x_scale)
    grid_dep_launch();
    if (a.fmt == MOE_FMT_NVFP4 && tid == 0) a.x_scale[t] = gs;
    const int S = fmt_sf_atoms(a.fmt);
    if (batched) {
        if (tid == 0) {
            s_rows[0] = t;
            s_sfb[0] = sf_row_base(t, S, fmt_k_stages(a.fmt, a.H));
        }
    } else if (tid < a.k) {
        const int s = t * a.k + tid, e = s_exp[tid];
        const int r = e >= 0 && e < a.E ? a.wbase[s / chunk * a.E + e] + s_rank[tid] : -1;
        a.inv[s] = r;
        s_rows[tid] = r;
        s_sfb[tid] = r >= 0 ? sf_row_base(r, S, fmt_k_stages(a.fmt, a.H)) : 0;
        if (r >= 0) a.src[r] = s;  // the routing kernel wrote the padding rows
    }
    __syncthreads();
    const int k = batched ? 1 : a.k;

#pragma unroll
    for (int i = 0; i < MAXC; ++i) {
        const int c = tid + i * NT;
        if (i * NT >= nchunks) break;  // uniform across the CTA
        const bool in = c < nchunks;
        float f[8];
        bf16x8_to_f32(v[i], f);
        if (a.fmt == MOE_FMT_BF16) {
            if (in)
                for (int j = 0; j < k; ++j) {
                    const int r = s_rows[j];
                    if (r >= 0) reinterpret_cast<uint4*>(a.xq + (int64_t)r * a.H * 2)[c] = v[i];
                }
        } else if (a.fmt == MOE_FMT_MXFP4) {
            // a 1x32 block is 4 neighbouring threads: exponent from the block amax, then
            // E2M1 codes of x * 2^-e, 8 codes (4 bytes) per thread
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const int ex = ue8m0_exponent_fp4(amax);
            const float sc = pow2f(-ex);  // ex in [-127, 127]
            uint32_t word = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) word |= cvt_e2m1x2(f[2 * j] * sc, f[2 * j + 1] * sc) << (8 * j);
            if (in)
                for (int j = 0; j < k; ++j) {
                    const int r = s_rows[j];
                    if (r < 0) continue;
                    reinterpret_cast<uint32_t*>(a.xq + (int64_t)r * (a.H / 2))[c] = word;
                    if ((c & 3) == 0) a.xsf[sf_byte(s_sfb[j], c / 4)] = (uint8_t)(ex + 127);
                }
        } else if (a.fmt == MOE_FMT_MXFP8) {
            const int ex = mxfp8_block_exponent(f);
            const uint2 codes = mxfp8_chunk(f, ex);
            if (in)
                for (int j = 0; j < k; ++j) {
                    const int r = s_rows[j];
                    if (r < 0) continue;
                    reinterpret_cast<uint2*>(a.xq + (int64_t)r * a.H)[c] = codes;
                    if ((c & 3) == 0) a.xsf[sf_byte(s_sfb[j], c / 4)] = (uint8_t)(ex + 127);
                }
        } else {
            float amax = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            const uint32_t sb = cvt_e4m3x2(__fdiv_rn(amax, __fmul_rn(gs, 6.0f)), 0.0f) & 0xFF;
            const float eff = __fmul_rn(e4m3_to_f32(sb), gs);
            uint32_t word = 0;
            if (eff > 0.0f) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    word |= cvt_e2m1x2(__fdiv_rn(f[2 * j], eff), __fdiv_rn(f[2 * j + 1], eff)) << (8 * j);
            }
            if (in)
                for (int j = 0; j < k; ++j) {
                    const int r = s_rows[j];
                    if (r < 0) continue;
                    reinterpret_cast<uint32_t*>(a.xq + (int64_t)r * (a.H / 2))[c] = word;
                    if ((c & 1) == 0) a.xsf[sf_byte(s_sfb[j], c / 2)] = (uint8_t)sb;
                }
        }
        // unpermuted copy for the shared expert
        if (batched) {
        } else if (a.shared_fmt == MOE_FMT_BF16) {
            if (in) reinterpret_cast<uint4*>(a.sxq + (int64_t)t * a.H * 2)[c] = v[i];
        } else if (a.shared_fmt == MOE_FMT_MXFP8) {
            const int ex = mxfp8_block_exponent(f);
            const uint2 codes = mxfp8_chunk(f, ex);
            if (in) {
                reinterpret_cast<uint2*>(a.sxq + (int64_t)t * a.H)[c] = codes;
                if ((c & 3) == 0)
                    a.sxsf[act_sf_offset(t, c / 4, 1, fmt_k_stages(MOE_FMT_MXFP8, a.H))] = (uint8_t)(ex + 127);
            }
        }
    }
    if (batched) __syncthreads();  // the next row reuses the shared arrays
}

template <int MAXC, int NT, int MIN_CTAS>
__global__ void __launch_bounds__(NT, MIN_CTAS) dispatch_kernel(const DispatchArgs a) {
    if (!a.batch_counts) {
        dispatch_one<MAXC, NT>(a, blockIdx.x, false);
        return;
    }
    // batched layout: the used rows, numbered 0 .. batch_prefix[E) in expert order, strided
    // over the grid; used row i is row e * M + (i - batch_prefix[e]) of the expert e with
    // batch_prefix[e] <= i < batch_prefix[e + 1]
    grid_dep_wait();  // the planning kernel has written batch_prefix
    grid_dep_launch();
    const int used = a.batch_prefix[a.E];
    for (int i = blockIdx.x; i < used; i += gridDim.x) {
        int lo = 0, hi = a.E;  // batch_prefix[lo] <= i < batch_prefix[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) / 2;
            if (a.batch_prefix[mid] <= i)
                lo = mid;
            else
                hi = mid;
        }
        dispatch_one<MAXC, NT>(a, lo * a.batch_M + (i - a.batch_prefix[lo]), true);
    }
}

cudaError_t launch_dispatch(const DispatchArgs& a, cudaStream_t st, bool pdl) {
    LaunchAttrs at(pdl);
    const int grid = a.batch_counts ? (a.T < 2048 ? a.T : 2048) : a.T;
    if (a.H <= DISPATCH_SMALL_CHUNKS * DISPATCH_NARROW_THREADS * 8 && grid >= DISPATCH_NARROW_MIN_TOKENS) {
        cudaLaunchConfig_t cfg = at.config(dim3(grid), dim3(DISPATCH_NARROW_THREADS), 0, st);
        return cudaLaunchKernelEx(
            &cfg, dispatch_kernel<DISPATCH_SMALL_CHUNKS, DISPATCH_NARROW_THREADS, DISPATCH_NARROW_MIN_CTAS>, a);
    }
    cudaLaunchConfig_t cfg = at.config(dim3(grid), dim3(DISPATCH_THREADS), 0, st);
    if (a.H <= DISPATCH_SMALL_CHUNKS * DISPATCH_THREADS * 8)
        return cudaLaunchKernelEx(&cfg, dispatch_kernel<DISPATCH_SMALL_CHUNKS, DISPATCH_THREADS, DISPATCH_SMALL_MIN_CTAS>,
                                  a);
    return cudaLaunchKernelEx(&cfg, dispatch_kernel<DISPATCH_MAX_CHUNKS, DISPATCH_THREADS, 3>, a);
}

}  // namespace moe
