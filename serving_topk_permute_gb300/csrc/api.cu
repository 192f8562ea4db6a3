// api.cu -- the C ABI of libmoe.so (include/moe.h): configuration checks, workspace
// layout, TMA tensor maps, and the stream-ordered launch sequence of moe_forward:
//   route -> dispatch quantisation -> L1 GEMM (SwiGLU + requant) -> L2 GEMM
//   [-> shared L1 -> shared L2] -> combine (+ shared) (+ RMSNorm).
#include <cudaTypedefs.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <new>

#include "common.cuh"
#include "kernels.h"

using namespace moe;

namespace {

constexpr int MAX_EXPERTS = 512;
constexpr int MAX_TOP_K = 32;
constexpr int MAX_HIDDEN = 16384;
constexpr int64_t REGION_ALIGN = 1024;
constexpr unsigned long long DEFAULT_TIMEOUT_NS = 2000000000ull;  // 2 s per bounded wait

struct Dims {
    int E, H, I, k, fmt, Is, sfmt;
};

Dims dims_of(const moe_config_t& c) {
    return Dims{c.num_experts, c.hidden, c.inter, c.top_k, c.format, c.shared_inter, c.shared_format};
}

int validate(const moe_config_t* c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->format != MOE_FMT_BF16 && c->format != MOE_FMT_MXFP8 && c->format != MOE_FMT_NVFP4 &&
        c->format != MOE_FMT_MXFP4)
        return MOE_ERR_UNSUPPORTED;
    if (c->activation != MOE_ACT_SWIGLU) return MOE_ERR_UNSUPPORTED;
    if (c->num_experts < 1 || c->num_experts > MAX_EXPERTS) return MOE_ERR_INVALID_ARG;
    if (c->top_k < 1 || c->top_k > c->num_experts || c->top_k > MAX_TOP_K) return MOE_ERR_INVALID_ARG;
    if (c->max_tokens < 1) return MOE_ERR_INVALID_ARG;
    if (c->hidden < 128 || c->inter < 128 || c->hidden % 128 || c->inter % 128) return MOE_ERR_INVALID_ARG;
    if (c->hidden > MAX_HIDDEN) return MOE_ERR_INVALID_ARG;
    if ((c->format == MOE_FMT_NVFP4 || c->format == MOE_FMT_MXFP4) && (c->hidden % 256 || c->inter % 256))
        return MOE_ERR_INVALID_ARG;  // a 128-byte K stage holds 256 four-bit elements
    if (!isfinite(c->act_alpha) || !isfinite(c->act_beta)) return MOE_ERR_INVALID_ARG;
    if (c->act_has_clamp && !(c->act_clamp >= 0.0f)) return MOE_ERR_INVALID_ARG;
    if (c->shared_inter < 0 || c->shared_inter % 128) return MOE_ERR_INVALID_ARG;
    if (c->shared_inter > 0) {
        if (c->shared_format != MOE_FMT_BF16 && c->shared_format != MOE_FMT_MXFP8) return MOE_ERR_UNSUPPORTED;
        if (c->shared_format == MOE_FMT_BF16 && (c->hidden % 256 || c->shared_inter % 256))
            return MOE_ERR_INVALID_ARG;
    }
    if (c->post_norm != 0 && c->post_norm != 1) return MOE_ERR_INVALID_ARG;
    if (!isfinite(c->norm_eps) || c->norm_eps < 0.0f) return MOE_ERR_INVALID_ARG;
    const int64_t R = (int64_t)c->max_tokens * c->top_k;
    if (R + (int64_t)c->num_experts * BM >= (int64_t)1 << 30) return MOE_ERR_INVALID_ARG;  // int32 row indices
    return MOE_OK;
}

// ------------------------------------------------------------------ GEMM variant per call
// The GEMMs run on CTA pairs (256 x 256 tiles, routed segments padded to 256 rows)
// only with MOE_FLAG_CTA_PAIR. Measured on GB300, pairs match single CTAs on the
// dense shared expert (0.127 vs 0.125 ms for its L1 at T=4096) and lose on routed
// prefill (L1 2.35 vs 2.14 ms), where 256-row padding adds MMA work; so single
// CTAs (128-row segments) are the default.
bool use_pair(const moe_config_t& c, int64_t rows_per_expert) {
    (void)rows_per_expert;
    if (c.flags & MOE_FLAG_CTA_SINGLE) return false;
    return (c.flags & MOE_FLAG_CTA_PAIR) != 0;
}

int64_t routed_rows_per_expert(const moe_config_t& c, int T) {
    return ceil_div((int64_t)T * c.top_k, c.num_experts);
}

int block_m_for(const moe_config_t& c, int T) { return use_pair(c, routed_rows_per_expert(c, T)) ? 2 * BM : BM; }

// ------------------------------------------------------------------ workspace layout
enum Region {
    R_ERR, R_META, R_CNT, R_OFF, R_TILE_EXPERT, R_SRC, R_INV, R_XSCALE, R_XQ, R_XSF, R_HQ, R_HSF, R_Y, R_HDBG,
    R_SXQ, R_SXSF, R_SHQ, R_SHSF, R_SY, R_SCHED, R_WBASE, R_COUNT
};

struct Layout {
    int64_t off[R_COUNT];
    int64_t size[R_COUNT];
    int64_t total;
    int64_t m_pad_max, m_tiles_max, t_pad;
};

Layout layout_of(const moe_config_t& c, int T) {
    Layout L{};
    const Dims d = dims_of(c);
    const int64_t R = (int64_t)T * d.k;
    const int bm = block_m_for(c, T);
    L.m_pad_max = align_up(R + (int64_t)d.E * (bm - 1), bm);
    if (L.m_pad_max == 0) L.m_pad_max = bm;
    L.m_tiles_max = L.m_pad_max / BM;
    L.t_pad = align_up(T > 0 ? T : 1, 2 * BM);
    const int S = fmt_sf_atoms(d.fmt);
    const int64_t nks_h = fmt_k_stages(d.fmt, d.H), nks_i = fmt_k_stages(d.fmt, d.I);
    int64_t sz[R_COUNT] = {};
    sz[R_ERR] = 16;
    sz[R_META] = 16;
    sz[R_CNT] = 4 * d.E;
    sz[R_OFF] = 4 * (d.E + 1);
    sz[R_TILE_EXPERT] = 4 * L.m_tiles_max;
    sz[R_SRC] = 4 * L.m_pad_max;
    sz[R_INV] = 4 * R;
    sz[R_XSCALE] = 4 * (int64_t)T;
    sz[R_XQ] = L.m_pad_max * fmt_row_bytes(d.fmt, d.H);
    sz[R_XSF] = L.m_tiles_max * nks_h * S * ATOM_BYTES;
    sz[R_HQ] = L.m_pad_max * fmt_row_bytes(d.fmt, d.I);
    sz[R_HSF] = L.m_tiles_max * nks_i * S * ATOM_BYTES;
    sz[R_Y] = L.m_pad_max * d.H * 2;
    sz[R_HDBG] = (c.flags & MOE_FLAG_DEBUG_H) ? L.m_pad_max * d.I * 4 : 0;
    if (d.Is > 0) {
        const int Ss = fmt_sf_atoms(d.sfmt);
        sz[R_SXQ] = L.t_pad * fmt_row_bytes(d.sfmt, d.H);
        sz[R_SXSF] = (L.t_pad / BM) * fmt_k_stages(d.sfmt, d.H) * Ss * ATOM_BYTES;
        sz[R_SHQ] = L.t_pad * fmt_row_bytes(d.sfmt, d.Is);
        sz[R_SHSF] = (L.t_pad / BM) * fmt_k_stages(d.sfmt, d.Is) * Ss * ATOM_BYTES;
        sz[R_SY] = L.t_pad * d.H * 2;
    }
    // schedule counters of the one-kernel GEMM: routed (counter, done[m_tiles_max]),
    // then shared (counter, done[t_pad / 128]); zeroed by the routing kernel
    sz[R_SCHED] = 4 * (2 + L.m_tiles_max + L.t_pad / BM);
    sz[R_WBASE] = 4 * ROUTE_WARPS * d.E;  // each routing chunk's first row in each expert
    int64_t o = 0;
    for (int r = 0; r < R_COUNT; ++r) {
        L.off[r] = o;
        L.size[r] = sz[r];
        o += align_up(sz[r], REGION_ALIGN);
    }
    L.total = o;
    return L;
}

// ------------------------------------------------------------------ TMA descriptors
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

bool get_encode() {
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode != nullptr;
}

// rows of row_bytes bytes, loaded as 128-byte x box_rows tiles with 128-byte swizzle
bool map_2d(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows) {
    cuuint64_t dims[2] = {row_bytes, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {(cuuint32_t)BK_BYTES, box_rows};
    cuuint32_t es[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [E][N][row_bytes] weights, loaded as 128-byte x bn-row tiles of one expert
bool map_3d(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t N, uint64_t E, uint32_t bn) {
    cuuint64_t dims[3] = {row_bytes, N, E};
    cuuint64_t strides[2] = {row_bytes, row_bytes * N};
    cuuint32_t box[3] = {(cuuint32_t)BK_BYTES, bn, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// an array of 512-byte scale atoms as a 2-D uint32 tensor [atoms][128], loaded box_atoms at a time
bool map_atoms(CUtensorMap* m, const void* base, uint64_t atoms, uint32_t box_atoms) {
    cuuint64_t dims[2] = {ATOM_BYTES / 4, atoms};
    cuuint64_t strides[1] = {ATOM_BYTES};
    cuuint32_t box[2] = {ATOM_BYTES / 4, box_atoms};
    cuuint32_t es[2] = {1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 255u) == 0; }
// every pointer a weight set carries is 256-byte aligned (null ones are checked elsewhere)
bool weights_aligned(const moe_weights_t* w) {
    for (const void* p : {(const void*)w->w13, (const void*)w->w13_sf, (const void*)w->w13_gs, (const void*)w->w2,
                          (const void*)w->w2_sf, (const void*)w->w2_gs})
        if (p && !aligned(p)) return false;
    return true;
}

}  // namespace

struct moe_plan_s {
    moe_config_t cfg;
    int device;
    int num_sms;
    unsigned long long timeout_ns;
    bool timing = false;
    bool pdl = true;  // programmatic dependent launch between the forward's kernels
    cudaEvent_t ev[2 * MOE_NUM_KERNELS] = {};
    bool ran[MOE_NUM_KERNELS] = {};
};

namespace {
// brackets one kernel launch with the plan's timing events (when enabled)
struct KernelTimer {
    moe_plan_s* p;
    int id;
    cudaStream_t st;
    KernelTimer(moe_plan_s* p_, int id_, cudaStream_t st_) : p(p_), id(id_), st(st_) {
        if (p->timing) {
            cudaEventRecord(p->ev[2 * id], st);
            p->ran[id] = true;
        }
    }
    ~KernelTimer() {
        if (p->timing) cudaEventRecord(p->ev[2 * id + 1], st);
    }
};
}  // namespace

// a failed runtime call is reported as MOE_ERR_CUDA and cleared from the runtime's
// last-error state, so that it does not surface in the caller's next CUDA call
#define CUDA_TRY(x)                      \
    do {                                 \
        if ((x) != cudaSuccess) {        \
            (void)cudaGetLastError();    \
            return MOE_ERR_CUDA;         \
        }                                \
    } while (0)

extern "C" {

int moe_config_validate(const moe_config_t* cfg) { return validate(cfg); }

int moe_plan(const moe_config_t* cfg, moe_plan_t* out) {
    if (!out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    const int v = validate(cfg);
    if (v != MOE_OK) return v;
    int dev = 0, major = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_UNSUPPORTED;
    CUDA_TRY(cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev));
    if (major != 10) return MOE_ERR_UNSUPPORTED;
    CUDA_TRY(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    if (!get_encode()) return MOE_ERR_CUDA;
    CUDA_TRY(route_prepare(MAX_EXPERTS));
    for (int f = MOE_FMT_BF16; f <= MOE_FMT_MXFP4; ++f) {
        CUDA_TRY(gemm_prepare(f));
        CUDA_TRY(gemm2_prepare(f));
        CUDA_TRY(fused_prepare(f));
    }
    CUDA_TRY(combine_prepare());
    moe_plan_s* p = new (std::nothrow) moe_plan_s;
    if (!p) return MOE_ERR_INVALID_ARG;
    p->cfg = *cfg;
    p->device = dev;
    p->num_sms = sms;
    p->timeout_ns = DEFAULT_TIMEOUT_NS;
    p->pdl = (cfg->flags & MOE_FLAG_SERIAL) == 0;
    *out = p;
    return MOE_OK;
}

int moe_plan_enable_timing(moe_plan_t plan, int32_t enable) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    if (enable && !plan->timing) {
        for (auto& e : plan->ev) CUDA_TRY(cudaEventCreate(&e));
        plan->timing = true;
    } else if (!enable && plan->timing) {
        for (auto& e : plan->ev) cudaEventDestroy(e);
        plan->timing = false;
    }
    return MOE_OK;
}

int moe_plan_set_wait_timeout(moe_plan_t plan, uint64_t timeout_ns) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    plan->timeout_ns = timeout_ns ? timeout_ns : DEFAULT_TIMEOUT_NS;
    return MOE_OK;
}

int moe_plan_kernel_times(moe_plan_t plan, float* ms, int32_t count) {
    if (!plan || !ms || count < MOE_NUM_KERNELS || !plan->timing) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < MOE_NUM_KERNELS; ++i) {
        ms[i] = 0.0f;
        if (!plan->ran[i]) continue;
        CUDA_TRY(cudaEventSynchronize(plan->ev[2 * i + 1]));
        CUDA_TRY(cudaEventElapsedTime(&ms[i], plan->ev[2 * i], plan->ev[2 * i + 1]));
    }
    return MOE_OK;
}

int moe_plan_destroy(moe_plan_t plan) {
    if (plan) moe_plan_enable_timing(plan, 0);
    delete plan;
    return MOE_OK;
}

int moe_plan_block_m(moe_plan_t plan, int32_t num_tokens, int32_t* block_m) {
    if (!plan || !block_m || num_tokens < 0) return MOE_ERR_INVALID_ARG;
    *block_m = block_m_for(plan->cfg, num_tokens);
    return MOE_OK;
}

int moe_config_workspace_size(const moe_config_t* cfg, int32_t num_tokens, size_t* bytes) {
    const int v = validate(cfg);
    if (v != MOE_OK) return v;
    if (!bytes || num_tokens < 0) return MOE_ERR_INVALID_ARG;
    if (num_tokens > cfg->max_tokens) return MOE_ERR_CAPACITY;
    *bytes = (size_t)layout_of(*cfg, num_tokens).total;
    return MOE_OK;
}

int moe_workspace_size(moe_plan_t plan, int32_t num_tokens, size_t* bytes) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    return moe_config_workspace_size(&plan->cfg, num_tokens, bytes);
}

int moe_workspace_region(moe_plan_t plan, int32_t num_tokens, int32_t which, size_t* offset, size_t* bytes) {
    if (!plan || !offset || !bytes || num_tokens < 0) return MOE_ERR_INVALID_ARG;
    static const int map[] = {R_CNT, R_OFF, R_SRC, R_INV, R_XQ, R_XSF, R_XSCALE, R_HQ, R_HSF, R_HDBG, R_Y, R_META, R_SY};
    if (which < 0 || which >= (int)(sizeof(map) / sizeof(map[0]))) return MOE_ERR_INVALID_ARG;
    const Layout L = layout_of(plan->cfg, num_tokens);
    *offset = (size_t)L.off[map[which]];
    *bytes = (size_t)L.size[map[which]];
    return MOE_OK;
}

static int64_t weight_bytes(const moe_config_t& c, int which) {
    const Dims d = dims_of(c);
    const bool shared = which >= MOE_SHARED_W13 && which <= MOE_SHARED_W2_SF;
    const int fmt = shared ? d.sfmt : d.fmt;
    const int64_t E = shared ? 1 : d.E, I = shared ? d.Is : d.I, H = d.H;
    if (shared && d.Is == 0) return 0;
    const int S = fmt_sf_atoms(fmt);
    switch (which) {
        case MOE_W13:
        case MOE_SHARED_W13: return E * 2 * I * fmt_row_bytes(fmt, H);
        case MOE_W2:
        case MOE_SHARED_W2: return E * H * fmt_row_bytes(fmt, I);
        case MOE_W13_SF:
        case MOE_SHARED_W13_SF: return E * fmt_k_stages(fmt, H) * wt_sf_blocks(2 * I) * S * ATOM_BYTES;
        case MOE_W2_SF:
        case MOE_SHARED_W2_SF: return E * fmt_k_stages(fmt, I) * wt_sf_blocks(H) * S * ATOM_BYTES;
        case MOE_W13_GS:
        case MOE_W2_GS: return d.fmt == MOE_FMT_NVFP4 ? 4 * E : 0;
        default: return -1;
    }
}

int moe_weight_layout_size(moe_plan_t plan, int32_t which, size_t* bytes) {
    if (!plan || !bytes) return MOE_ERR_INVALID_ARG;
    const int64_t b = weight_bytes(plan->cfg, which);
    if (b < 0) return MOE_ERR_INVALID_ARG;
    *bytes = (size_t)b;
    return MOE_OK;
}

static int transform(const moe_config_t& c, int fmt, int E, int I, const moe_weights_t* src, moe_weights_t* dst,
                     bool gscales, cudaStream_t st) {
    const int H = c.hidden;
    if (!src || !dst || !src->w13 || !src->w2 || !dst->w13 || !dst->w2) return MOE_ERR_INVALID_ARG;
    if (!weights_aligned(src) || !weights_aligned(dst)) return MOE_ERR_INVALID_ARG;
    if (src->w13 == dst->w13 || src->w2 == dst->w2) return MOE_ERR_INVALID_ARG;
    const bool scaled = fmt != MOE_FMT_BF16;
    if (scaled && (!src->w13_sf || !src->w2_sf || !dst->w13_sf || !dst->w2_sf)) return MOE_ERR_INVALID_ARG;
    if (gscales && fmt == MOE_FMT_NVFP4 && (!src->w13_gs || !src->w2_gs || !dst->w13_gs || !dst->w2_gs))
        return MOE_ERR_INVALID_ARG;
    CUDA_TRY(launch_interleave_rows((const uint8_t*)src->w13, (uint8_t*)dst->w13, E, I, fmt_row_bytes(fmt, H), st));
    CUDA_TRY(cudaMemcpyAsync(dst->w2, src->w2, (size_t)E * H * fmt_row_bytes(fmt, I), cudaMemcpyDeviceToDevice, st));
    if (scaled) {
        CUDA_TRY(launch_pack_weight_sf((const uint8_t*)src->w13_sf, (uint8_t*)dst->w13_sf, fmt, E, 2 * I, H, true, I,
                                       st));
        CUDA_TRY(launch_pack_weight_sf((const uint8_t*)src->w2_sf, (uint8_t*)dst->w2_sf, fmt, E, H, I, false, I, st));
    }
    if (gscales && fmt == MOE_FMT_NVFP4) {
        CUDA_TRY(cudaMemcpyAsync(dst->w13_gs, src->w13_gs, 4 * (size_t)E, cudaMemcpyDeviceToDevice, st));
        CUDA_TRY(cudaMemcpyAsync(dst->w2_gs, src->w2_gs, 4 * (size_t)E, cudaMemcpyDeviceToDevice, st));
    }
    return MOE_OK;
}

int moe_transform_weights(moe_plan_t plan, const moe_weights_t* src, moe_weights_t* dst, void* stream) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    const moe_config_t& c = plan->cfg;
    return transform(c, c.format, c.num_experts, c.inter, src, dst, true, (cudaStream_t)stream);
}

int moe_transform_shared_weights(moe_plan_t plan, const moe_weights_t* src, moe_weights_t* dst, void* stream) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    const moe_config_t& c = plan->cfg;
    if (c.shared_inter == 0) return MOE_ERR_INVALID_ARG;
    return transform(c, c.shared_format, 1, c.shared_inter, src, dst, false, (cudaStream_t)stream);
}

// one expert MLP pass (L1 then L2) over row tiles of the given A buffers
// N-tile width. Measured on GB300 at every workload, 256-wide tiles (one accumulator,
// 4-stage ring) beat 128-wide tiles with double-buffered accumulators (6 stages): the
// narrower tile reloads the A tile twice as often per weight byte. So 256 unless
// MOE_FLAG_TILE_128 forces 128.
static int choose_bn(const moe_config_t& c, int64_t rows_per_expert) {
    (void)rows_per_expert;
    if (c.flags & MOE_FLAG_TILE_128) return 128;
    return 256;
}

// Batched layout: row-tile first rows and per-expert used-row counts (see BatchedDeepGemmExperts)
struct BatchRows {
    const int* tile_row;
    const int* counts;
    int rows_per_expert;
};

// one expert MLP pass; m_tiles_* count 128-row tiles on single CTAs, 256-row tiles on pairs.
// With 256-wide single-CTA tiles (the default), L1 and L2 run as one kernel (sched:
// its zeroed counters); otherwise as two.
static int run_mlp(moe_plan_s* p, int kid1, int fmt, int E, int I, int H, bool pair, const void* xq,
                   const uint8_t* xsf, int64_t rows,
                   const moe_weights_t* w, const int* m_tiles_dev, int m_tiles_host, int64_t m_tiles_max,
                   const int* tile_expert, const int* src, int m_valid, const float* x_scale, const float* a2,
                   uint8_t* hq, uint8_t* hsf, float* h_debug, __nv_bfloat16* y, int* err, bool activation,
                   uint32_t* sched, cudaStream_t st, const BatchRows* br = nullptr,
                   const int* seg_off = nullptr, const int* seg_cnt = nullptr, bool independent = false) {
    const moe_config_t& c = p->cfg;
    const int S = fmt_sf_atoms(fmt);
    const int bn = pair ? 2 * BM : choose_bn(c, 0);
    const uint32_t b_box = pair ? NBLK : bn;  // a CTA of a pair loads half of the 256 weight rows
    const bool fused = !pair && bn == 256 && sched && !(c.flags & MOE_FLAG_SPLIT_GEMM);
    CUtensorMap ta1, tb1, ta2, tb2, tsa1, tsb1, tsa2, tsb2, ta1s, ta2s;
    GemmArgs g{};
    g.m_tiles_dev = m_tiles_dev;
    g.m_tiles_host = m_tiles_host;
    g.tile_expert = tile_expert;
    g.src = src;
    g.m_valid = m_valid;
    g.seg_off = seg_off;
    g.seg_cnt = seg_cnt;
    if (br) {
        g.tile_row = br->tile_row;
        g.counts = br->counts;
        g.rows_per_expert = br->rows_per_expert;
    }
    g.top_k = c.top_k;
    g.err = err;
    g.timeout_ns = p->timeout_ns;
    g.act_alpha = activation ? c.act_alpha : 1.0f;
    g.act_beta = activation ? c.act_beta : 0.0f;
    g.act_clamp = c.act_clamp;
    g.act_has_clamp = activation ? c.act_has_clamp : 0;
    g.x_scale = x_scale;
    g.a2 = a2;
    g.hq = hq;
    g.hsf = hsf;
    g.I = I;
    g.h_nks = (int)fmt_k_stages(fmt, I);
    g.h_debug = h_debug;
    g.y = y;
    g.ldy = H;
    // L1: [rows, H] x w13[e]^T -> h [rows, I]
    GemmArgs g1 = g;
    g1.sfa = xsf;
    g1.sfb = (const uint8_t*)w->w13_sf;
    g1.nks = (int)fmt_k_stages(fmt, H);
    g1.n_tiles = (int)ceil_div(2 * I, bn);
    g1.sf_blocks = (int)wt_sf_blocks(2 * I);
    g1.N = 2 * I;
    g1.gscale = w->w13_gs;
    if (!map_2d(&ta1, xq, fmt_row_bytes(fmt, H), rows, BM)) return MOE_ERR_CUDA;
    if (!map_3d(&tb1, w->w13, fmt_row_bytes(fmt, H), 2 * (uint64_t)I, E, b_box)) return MOE_ERR_CUDA;
    // L2: h [rows, I] x w2[e]^T -> y [rows, H]
    GemmArgs g2 = g;
    g2.sfa = hsf;
    g2.sfb = (const uint8_t*)w->w2_sf;
    g2.nks = (int)fmt_k_stages(fmt, I);
    g2.n_tiles = (int)ceil_div(H, bn);
    g2.sf_blocks = (int)wt_sf_blocks(H);
    g2.N = H;
    g2.gscale = w->w2_gs;
    if (!map_2d(&ta2, hq, fmt_row_bytes(fmt, I), rows, BM)) return MOE_ERR_CUDA;
    if (!map_3d(&tb2, w->w2, fmt_row_bytes(fmt, I), H, E, b_box)) return MOE_ERR_CUDA;
    if (pair && S) {
        const uint32_t sfb_box = (uint32_t)S * (2 * BM / NBLK);
        if (!map_atoms(&tsa1, xsf, (uint64_t)(rows / BM) * g1.nks * S, S)) return MOE_ERR_CUDA;
        if (!map_atoms(&tsb1, w->w13_sf, (uint64_t)E * g1.nks * g1.sf_blocks * S, sfb_box)) return MOE_ERR_CUDA;
        if (!map_atoms(&tsa2, hsf, (uint64_t)(rows / BM) * g2.nks * S, S)) return MOE_ERR_CUDA;
        if (!map_atoms(&tsb2, w->w2_sf, (uint64_t)E * g2.nks * g2.sf_blocks * S, sfb_box)) return MOE_ERR_CUDA;
    }
    if (fused) {
        // the one-kernel GEMM loads mostly empty row tiles in smaller boxes
        if (!map_2d(&ta1s, xq, fmt_row_bytes(fmt, H), rows, A_BOX_ROWS)) return MOE_ERR_CUDA;
        if (!map_2d(&ta2s, hq, fmt_row_bytes(fmt, I), rows, A_BOX_ROWS)) return MOE_ERR_CUDA;
        FusedSched fs{sched, sched + 1, independent && p->pdl ? 1 : 0};
        const int64_t tiles = m_tiles_max * (g1.n_tiles + g2.n_tiles);
        const int grid = (int)std::min<int64_t>(p->num_sms, std::max<int64_t>(1, tiles));
        KernelTimer kt(p, kid1, st);
        CUDA_TRY(launch_fused_mlp(fmt, ta1, tb1, ta2, tb2, ta1s, ta2s, g1, g2, fs, grid, st, p->pdl));
        return MOE_OK;
    }
    auto launch = [&](bool l1, const GemmArgs& ga, int64_t tiles) {
        const CUtensorMap& ta = l1 ? ta1 : ta2;
        const CUtensorMap& tb = l1 ? tb1 : tb2;
        if (pair) {
            const int grid = 2 * (int)std::min<int64_t>(p->num_sms / 2, std::max<int64_t>(1, tiles));
            const CUtensorMap& tsa = S ? (l1 ? tsa1 : tsa2) : ta;
            const CUtensorMap& tsb = S ? (l1 ? tsb1 : tsb2) : tb;
            return launch_gemm2(fmt, l1, ta, tb, tsa, tsb, ga, grid, st, p->pdl);
        }
        const int grid = (int)std::min<int64_t>(p->num_sms, std::max<int64_t>(1, tiles));
        return launch_gemm(fmt, l1, bn, ta, tb, ga, grid, st, p->pdl);
    };
    {
        KernelTimer kt(p, kid1, st);
        CUDA_TRY(launch(true, g1, m_tiles_max * g1.n_tiles));
    }
    {
        KernelTimer kt(p, kid1 + 1, st);
        CUDA_TRY(launch(false, g2, m_tiles_max * g2.n_tiles));
    }
    return MOE_OK;
}

int moe_forward(moe_plan_t plan, int32_t T, const void* hidden, const int32_t* topk_ids, const float* topk_weights,
                const moe_weights_t* weights, const float* l2_act_scale, const moe_weights_t* shared,
                const float* norm_gamma, void* out, void* workspace, size_t workspace_bytes, void* stream) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    const moe_config_t& c = plan->cfg;
    const Dims d = dims_of(c);
    if (T < 0) return MOE_ERR_INVALID_ARG;
    if (T > c.max_tokens) return MOE_ERR_CAPACITY;
    if (T == 0) return MOE_OK;
    if (!hidden || !topk_ids || !topk_weights || !weights || !out || !workspace) return MOE_ERR_INVALID_ARG;
    if (!aligned(hidden) || !aligned(topk_ids) || !aligned(topk_weights) || !aligned(out) || !aligned(workspace))
        return MOE_ERR_INVALID_ARG;
    if (out == hidden) return MOE_ERR_INVALID_ARG;
    if (!weights->w13 || !weights->w2) return MOE_ERR_INVALID_ARG;
    if (d.fmt != MOE_FMT_BF16 && (!weights->w13_sf || !weights->w2_sf)) return MOE_ERR_INVALID_ARG;
    if (d.fmt == MOE_FMT_NVFP4 && (!weights->w13_gs || !weights->w2_gs || !l2_act_scale)) return MOE_ERR_INVALID_ARG;
    if (d.Is > 0 && (!shared || !shared->w13 || !shared->w2)) return MOE_ERR_INVALID_ARG;
    if (d.Is > 0 && d.sfmt != MOE_FMT_BF16 && (!shared->w13_sf || !shared->w2_sf)) return MOE_ERR_INVALID_ARG;
    if (c.post_norm && (!norm_gamma || !aligned(norm_gamma))) return MOE_ERR_INVALID_ARG;
    if (!weights_aligned(weights) || (d.Is > 0 && !weights_aligned(shared))) return MOE_ERR_INVALID_ARG;
    if (d.fmt == MOE_FMT_NVFP4 && !aligned(l2_act_scale)) return MOE_ERR_INVALID_ARG;
    const Layout L = layout_of(c, T);
    if (workspace_bytes < (size_t)L.total) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t* ws = (uint8_t*)workspace;
    auto R = [&](int r) { return ws + L.off[r]; };
    int* err = (int*)R(R_ERR);
    int* meta = (int*)R(R_META);
    const bool routed_pair = use_pair(c, routed_rows_per_expert(c, T));
    const int bm = routed_pair ? 2 * BM : BM;
    for (bool& r : plan->ran) r = false;  // the routing kernel zeroes the error word first

    {
        KernelTimer kt(plan, MOE_KERNEL_ROUTE, st);
        CUDA_TRY(launch_route(topk_ids, T, d.k, d.E, bm, (int*)R(R_CNT), (int*)R(R_OFF), (int*)R(R_SRC), (int*)R(R_INV),
                          (int*)R(R_TILE_EXPERT), meta, err, st, plan->pdl, (uint32_t*)R(R_SCHED),
                          (int)(L.size[R_SCHED] / 4), (int*)R(R_WBASE)));
    }
    DispatchArgs da{};
    da.x = (const uint16_t*)hidden;
    da.T = T;
    da.H = d.H;
    da.k = d.k;
    da.ids = topk_ids;
    da.E = d.E;
    da.wbase = (const int*)R(R_WBASE);
    da.inv = (int*)R(R_INV);
    da.src = (int*)R(R_SRC);
    da.fmt = d.fmt;
    da.xq = R(R_XQ);
    da.xsf = R(R_XSF);
    da.x_scale = (float*)R(R_XSCALE);
    da.shared_fmt = d.Is > 0 ? d.sfmt : -1;
    da.sxq = R(R_SXQ);
    da.sxsf = R(R_SXSF);
    {
        KernelTimer kt(plan, MOE_KERNEL_DISPATCH, st);
        CUDA_TRY(launch_dispatch(da, st, plan->pdl));
    }

    int rc = run_mlp(plan, MOE_KERNEL_L1, d.fmt, d.E, d.I, d.H, routed_pair, R(R_XQ), R(R_XSF), L.m_pad_max, weights,
                     meta + 1, 0, L.m_pad_max / bm,
                     (const int*)R(R_TILE_EXPERT), (const int*)R(R_SRC), 0, (const float*)R(R_XSCALE), l2_act_scale,
                     R(R_HQ), R(R_HSF), (c.flags & MOE_FLAG_DEBUG_H) ? (float*)R(R_HDBG) : nullptr,
                     (__nv_bfloat16*)R(R_Y), err, true, (uint32_t*)R(R_SCHED), st, nullptr, (const int*)R(R_OFF),
                     (const int*)R(R_CNT));
    if (rc != MOE_OK) return rc;
    if (d.Is > 0) {
        const bool shared_pair = use_pair(c, T);
        const int tiles = (int)(L.t_pad / (shared_pair ? 2 * BM : BM));
        rc = run_mlp(plan, MOE_KERNEL_SHARED_L1, d.sfmt, 1, d.Is, d.H, shared_pair, R(R_SXQ), R(R_SXSF), L.t_pad, shared, nullptr, tiles, tiles, nullptr,
                     nullptr, T, nullptr, nullptr, R(R_SHQ), R(R_SHSF), nullptr, (__nv_bfloat16*)R(R_SY), err, false,
                     (uint32_t*)R(R_SCHED) + 1 + L.m_tiles_max, st, nullptr, nullptr, nullptr,
                     /*independent: reads only dispatch's shared-expert rows, never the routed GEMMs' output*/ true);
        if (rc != MOE_OK) return rc;
    }
    CombineArgs ca{};
    ca.y = (const __nv_bfloat16*)R(R_Y);
    ca.inv = (const int*)R(R_INV);
    ca.w = topk_weights;
    ca.T = T;
    ca.k = d.k;
    ca.H = d.H;
    ca.ys = d.Is > 0 ? (const __nv_bfloat16*)R(R_SY) : nullptr;
    ca.gamma = c.post_norm ? norm_gamma : nullptr;
    ca.eps = c.norm_eps;
    ca.out = (__nv_bfloat16*)out;
    {
        KernelTimer kt(plan, MOE_KERNEL_COMBINE, st);
        CUDA_TRY(launch_combine(ca, st, plan->pdl));
    }
    return MOE_OK;
}

// ------------------------------------------------------------------ batched (masked) layout
namespace {
enum BRegion { B_ERR, B_META, B_TILE_EXPERT, B_TILE_ROW, B_ROW_PREFIX, B_XQ, B_XSF, B_XSCALE, B_HQ, B_HSF, B_SCHED,
               B_COUNT };
struct BLayout {
    int64_t off[B_COUNT];
    int64_t size[B_COUNT];
    int64_t total, rows, tiles;
};

BLayout batched_layout_of(const moe_config_t& c, int M) {
    BLayout L{};
    const Dims d = dims_of(c);
    L.rows = (int64_t)d.E * M;
    L.tiles = L.rows / BM;
    const int S = fmt_sf_atoms(d.fmt);
    int64_t sz[B_COUNT] = {};
    sz[B_ERR] = 16;  // first, at offset 0, as in moe_forward's workspace (moe_last_status reads it there)
    sz[B_META] = 16;
    sz[B_TILE_EXPERT] = 4 * L.tiles;
    sz[B_TILE_ROW] = 4 * L.tiles;
    sz[B_ROW_PREFIX] = 4 * (d.E + 1);
    sz[B_XQ] = L.rows * fmt_row_bytes(d.fmt, d.H);
    sz[B_XSF] = L.tiles * fmt_k_stages(d.fmt, d.H) * S * ATOM_BYTES;
    sz[B_XSCALE] = 4 * L.rows;
    sz[B_HQ] = L.rows * fmt_row_bytes(d.fmt, d.I);
    sz[B_HSF] = L.tiles * fmt_k_stages(d.fmt, d.I) * S * ATOM_BYTES;
    sz[B_SCHED] = 4 * (1 + L.tiles);  // the GEMM's tile counter and done[tiles]
    int64_t o = 0;
    for (int r = 0; r < B_COUNT; ++r) {
        L.off[r] = o;
        L.size[r] = sz[r];
        o += align_up(sz[r], REGION_ALIGN);
    }
    L.total = o;
    return L;
}

int batched_check(const moe_config_t& c, int32_t M) {
    if (M < BM || M % BM) return MOE_ERR_INVALID_ARG;
    if ((int64_t)c.num_experts * M >= ((int64_t)1 << 30)) return MOE_ERR_INVALID_ARG;  // int32 row indices
    if (c.flags & (MOE_FLAG_CTA_PAIR | MOE_FLAG_TILE_128 | MOE_FLAG_SPLIT_GEMM)) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}
}  // namespace

int moe_batched_workspace_size(moe_plan_t plan, int32_t max_tokens, size_t* bytes) {
    if (!plan || !bytes) return MOE_ERR_INVALID_ARG;
    const int v = batched_check(plan->cfg, max_tokens);
    if (v != MOE_OK) return v;
    *bytes = (size_t)batched_layout_of(plan->cfg, max_tokens).total;
    return MOE_OK;
}

int moe_forward_batched(moe_plan_t plan, int32_t max_tokens, const void* hidden, const int32_t* expert_num_tokens,
                        const moe_weights_t* weights, const float* l2_act_scale, void* out, void* workspace,
                        size_t workspace_bytes, void* stream) {
    if (!plan) return MOE_ERR_INVALID_ARG;
    const moe_config_t& c = plan->cfg;
    const Dims d = dims_of(c);
    const int v = batched_check(c, max_tokens);
    if (v != MOE_OK) return v;
    if (!hidden || !expert_num_tokens || !weights || !out || !workspace) return MOE_ERR_INVALID_ARG;
    if (!aligned(hidden) || !aligned(expert_num_tokens) || !aligned(out) || !aligned(workspace))
        return MOE_ERR_INVALID_ARG;
    if (out == hidden) return MOE_ERR_INVALID_ARG;
    if (!weights->w13 || !weights->w2) return MOE_ERR_INVALID_ARG;
    if (d.fmt != MOE_FMT_BF16 && (!weights->w13_sf || !weights->w2_sf)) return MOE_ERR_INVALID_ARG;
    if (d.fmt == MOE_FMT_NVFP4 && (!weights->w13_gs || !weights->w2_gs || !l2_act_scale)) return MOE_ERR_INVALID_ARG;
    if (!weights_aligned(weights) || (d.fmt == MOE_FMT_NVFP4 && !aligned(l2_act_scale))) return MOE_ERR_INVALID_ARG;
    const BLayout L = batched_layout_of(c, max_tokens);
    if (workspace_bytes < (size_t)L.total) return MOE_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    uint8_t* ws = (uint8_t*)workspace;
    auto R = [&](int r) { return ws + L.off[r]; };
    int* err = (int*)R(B_ERR);
    int* meta = (int*)R(B_META);
    uint32_t* sched = (uint32_t*)R(B_SCHED);
    for (bool& r : plan->ran) r = false;
    {
        KernelTimer kt(plan, MOE_KERNEL_ROUTE, st);
        CUDA_TRY(launch_batched_plan(expert_num_tokens, d.E, max_tokens, (int*)R(B_TILE_EXPERT), (int*)R(B_TILE_ROW),
                                     (int*)R(B_ROW_PREFIX), meta, err, sched, (int)(1 + L.tiles), st, plan->pdl));
    }
    DispatchArgs da{};
    da.x = (const uint16_t*)hidden;
    da.T = (int)L.rows;
    da.H = d.H;
    da.k = 1;
    da.E = d.E;
    da.fmt = d.fmt;
    da.xq = R(B_XQ);
    da.xsf = R(B_XSF);
    da.x_scale = (float*)R(B_XSCALE);
    da.shared_fmt = -1;
    da.batch_counts = expert_num_tokens;
    da.batch_prefix = (const int*)R(B_ROW_PREFIX);
    da.batch_M = max_tokens;
    {
        KernelTimer kt(plan, MOE_KERNEL_DISPATCH, st);
        CUDA_TRY(launch_dispatch(da, st, plan->pdl));
    }
    const BatchRows br{(const int*)R(B_TILE_ROW), expert_num_tokens, max_tokens};
    return run_mlp(plan, MOE_KERNEL_L1, d.fmt, d.E, d.I, d.H, false, R(B_XQ), R(B_XSF), L.rows, weights, meta + 1, 0,
                   L.tiles, (const int*)R(B_TILE_EXPERT), nullptr, 0, (const float*)R(B_XSCALE), l2_act_scale,
                   R(B_HQ), R(B_HSF), nullptr, (__nv_bfloat16*)out, err, true, sched, st, &br);
}

int moe_last_status(moe_plan_t plan, void* workspace, void* stream, int32_t* status) {
    if (!plan || !workspace || !status) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    int v = 0;
    CUDA_TRY(cudaMemcpyAsync(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost, st));
    CUDA_TRY(cudaStreamSynchronize(st));
    CUDA_TRY(cudaMemsetAsync(workspace, 0, sizeof(int), st));
    CUDA_TRY(cudaStreamSynchronize(st));
    *status = v;
    return MOE_OK;
}

const char* moe_error_string(int32_t status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, or unsupported shape)";
        case MOE_ERR_UNSUPPORTED: return "unsupported device, format or activation";
        case MOE_ERR_CAPACITY: return "num_tokens exceeds max_tokens";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA runtime error";
        case MOE_ERR_BAD_EXPERT_ID: return "expert id outside [-1, num_experts)";
        case MOE_ERR_TIMEOUT: return "a bounded device-side wait timed out";
        default: return "unknown status";
    }
}

}  // extern "C"
