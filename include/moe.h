/*
 * moe.h -- C ABI of the GB300 routed-expert MoE layer forward (libmoe.so).
 *
 * The layer (vllm.model_executor.layers.fused_moe.deep_gemm_mega_moe,
 * DeepGemmMegaMoEExperts; the unfused steps of vllm.model_executor.layers.
 * fused_moe, DeepGemmExperts.apply):
 *
 *   top-k permute (dispatch) -> L1 grouped GEMM on w13 (gate rows, then up
 *   rows) with SwiGLU and the requantisation of the L2 input in its
 *   epilogue -> L2 grouped GEMM on w2 -> top-k-weighted combine
 *   (+ optional shared expert) (-> optional post-expert RMSNorm) -> bf16.
 *
 * Formats: BF16; MXFP8 (E4M3 values, one UE8M0 scale per 1x32 K-block);
 * NVFP4 (E2M1 values packed two per byte, element 2i in the low nibble, one
 * E4M3 scale per 1x16 block, a per-expert FP32 global scale, and a per-token
 * FP32 dispatch scale computed by the layer).
 *
 * Conventions for every call:
 *   - Return value: MOE_OK (0) or one of the MOE_ERR_* codes below; on error
 *     nothing was launched unless the code is MOE_ERR_CUDA.
 *   - Pointers documented as "device" are device pointers owned by the
 *     caller; the library never frees them and never allocates device memory
 *     in moe_forward / moe_transform_weights (the caller passes a workspace).
 *   - GPU work is enqueued on the given stream and is asynchronous; inputs
 *     must stay valid until the stream reaches the work.
 *   - Every device pointer must be 256-byte aligned (MOE_ERR_INVALID_ARG).
 *   - moe_forward's hidden, topk_ids, topk_weights, norm_gamma and out may
 *     also be pinned host memory mapped into the device address space
 *     (cudaHostAlloc / cudaMallocHost under unified addressing): the routing,
 *     dispatch and combine kernels, the only ones that touch them, then read
 *     the inputs and write the output over the host link, with no separate
 *     copy. Weights and the workspace must be device memory.
 *   - Bad expert ids and bounded-wait timeouts found on the device are
 *     recorded in an error word in the workspace; read it with
 *     moe_last_status (which synchronises the stream).
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status codes */
#define MOE_OK                 0
#define MOE_ERR_INVALID_ARG    1   /* null / misaligned pointer, bad shape (the pages' ValueError) */
#define MOE_ERR_UNSUPPORTED    2   /* device arch / format / activation (the pages' NotImplementedError) */
#define MOE_ERR_CAPACITY       3   /* num_tokens > max_tokens (DeepGemmMegaMoEExperts.forward) */
#define MOE_ERR_WORKSPACE      4   /* workspace smaller than moe_workspace_size */
#define MOE_ERR_CUDA           5   /* a CUDA runtime call failed */
#define MOE_ERR_BAD_EXPERT_ID  6   /* a topk id outside [-1, E) was seen on the device */
#define MOE_ERR_TIMEOUT        7   /* a bounded device-side wait ran out */

/* ---------------------------------------------------------------- enums */
#define MOE_FMT_BF16   0
#define MOE_FMT_MXFP8  1
#define MOE_FMT_NVFP4  2
#define MOE_FMT_MXFP4  3   /* E2M1 codes, one UE8M0 scale per 1x32 block (weights, dispatch, L2 input) */

#define MOE_ACT_SWIGLU 0

#define MOE_FLAG_DEBUG_H  1u       /* also keep the fp32 L1 epilogue output h in the workspace */
#define MOE_FLAG_TILE_128 2u       /* 128-wide GEMM tiles with double-buffered accumulators */
#define MOE_FLAG_TILE_256 4u       /* 256-wide GEMM tiles (the default) */
#define MOE_FLAG_CTA_PAIR 8u       /* run the GEMMs on CTA pairs (256 x 256 tiles, BLOCK_M 256) */
#define MOE_FLAG_CTA_SINGLE 16u    /* run the GEMMs on single CTAs (the default) */
#define MOE_FLAG_SPLIT_GEMM 64u    /* run L1 and L2 as two kernels (by default, with 256-wide single-CTA tiles,
                                      one persistent kernel takes all L1 tiles, then all L2 tiles, from one
                                      counter, each L2 tile starting once its rows' L1 tiles are done) */
#define MOE_FLAG_SERIAL   32u      /* launch each kernel only after the previous one has finished (by default
                                      a kernel's set-up overlaps the previous kernel's tail: programmatic
                                      dependent launch, with every read of the previous output after the wait) */

/* ---------------------------------------------------------------- config / plan */

/*
 * Layer configuration (DeepGemmMegaMoEExperts constructor arguments:
 * num_experts, top_k, hidden_size, intermediate_size, activation,
 * weight_format, shared experts, max tokens).
 *
 * Validation (moe_config_validate, moe_plan):
 *   hidden, inter multiples of 128 (check_deep_gemm_mega_moe_supported);
 *   multiples of 256 for NVFP4 routed weights or a BF16 shared expert
 *   (vllm.models.muse_spark.nvidia.mega_moe, MuseSparkMegaMoEExperts);
 *   1 <= top_k <= num_experts <= 512; max_tokens >= 1;
 *   activation: finite alpha/beta, clamp >= 0 when has_clamp
 *   (MegaMoEActivation.__post_init__);
 *   shared_inter 0 (none) or a multiple of 128, shared_format BF16 or MXFP8;
 *   post_norm 0 or 1, norm_eps finite and >= 0; top_k <= 32; hidden <= 16384.
 */
typedef struct moe_config {
    int32_t num_experts;     /* E */
    int32_t hidden;          /* H */
    int32_t inter;           /* I */
    int32_t top_k;           /* k */
    int32_t max_tokens;      /* capacity: moe_forward rejects num_tokens > max_tokens */
    int32_t format;          /* MOE_FMT_* of the routed experts and of the L2 input */
    int32_t activation;      /* MOE_ACT_SWIGLU */
    float   act_alpha;       /* gate * sigmoid(alpha * gate) * (up + beta); default 1 */
    float   act_beta;        /* default 0 */
    float   act_clamp;       /* gate <= clamp, |up| <= clamp, used when act_has_clamp */
    int32_t act_has_clamp;
    int32_t shared_inter;    /* I_s of the shared expert, 0 = none */
    int32_t shared_format;   /* MOE_FMT_BF16 or MOE_FMT_MXFP8 */
    int32_t post_norm;       /* 1: RMSNorm of (routed + shared) with gamma applied verbatim */
    float   norm_eps;
    uint32_t flags;          /* MOE_FLAG_* */
} moe_config_t;

typedef struct moe_plan_s* moe_plan_t;

/* Host-only validation of a configuration (no CUDA call). */
int moe_config_validate(const moe_config_t* cfg);

/*
 * Create a plan for the current CUDA device. Validates cfg, checks the device
 * is compute capability 10.x (sm_103a code; MOE_ERR_UNSUPPORTED otherwise)
 * and caches per-device kernel attributes. *out is owned by the library:
 * release it with moe_plan_destroy.
 */
int moe_plan(const moe_config_t* cfg, moe_plan_t* out);
int moe_plan_destroy(moe_plan_t plan);

/*
 * BLOCK_M the routing pads each expert segment to for num_tokens tokens
 * (DeepGemmMegaMoEExperts.get_block_m; the pages' rule is inside a closed
 * library). Ours: 128, the MMA tile height of one CTA; 256 when the plan runs
 * its GEMMs on CTA pairs (MOE_FLAG_CTA_PAIR). Deterministic in (plan, num_tokens).
 */
int moe_plan_block_m(moe_plan_t plan, int32_t num_tokens, int32_t* block_m);

/*
 * Bytes of the caller-allocated workspace moe_forward needs for num_tokens
 * tokens (it replaces the pages' symmetric staging buffer,
 * DeepGemmMegaMoEExperts.get_symm_buffer). Host-only; the _cfg form needs no
 * plan and no device.
 */
int moe_workspace_size(moe_plan_t plan, int32_t num_tokens, size_t* bytes);
int moe_config_workspace_size(const moe_config_t* cfg, int32_t num_tokens, size_t* bytes);

/* ---------------------------------------------------------------- weights */

/*
 * Expert weights. Checkpoint layout (src of moe_transform_weights), E experts:
 *   w13      [E, 2I, H/vpe]  gate rows 0..I-1, then up rows (w1 then w3)
 *   w13_sf   [E, 2I, H/g]    u8 block scales, row-major (MXFP8: UE8M0, g=32;
 *                            NVFP4: E4M3, g=16; BF16: unused, NULL)
 *   w2       [E, H, I/vpe]
 *   w2_sf    [E, H, I/g]
 *   w13_gs   [E] fp32        NVFP4 global scale of w13[e] (the L1 alpha); else NULL
 *   w2_gs    [E] fp32        NVFP4 global scale of w2[e]; else NULL
 * vpe (values per byte-element): 1 for BF16 (2-byte elements) and MXFP8, 2 for NVFP4.
 *
 * Kernel layout (dst of moe_transform_weights, what moe_forward reads):
 *   w13  [E, 2I, H/vpe] with rows interleaved per 128-row block: kernel row
 *        128*b + 64*half + r holds checkpoint row half*I + 64*b + r
 *        (half 0 = gate, 1 = up; 0 <= r < 64), so every 128-row block holds 64
 *        gate and the matching 64 up rows (the pages interleave by 8,
 *        DeepGemmMegaMoEExperts._kernel_layout_shard).
 *   w2   unchanged.
 *   *_sf scale-factor atoms for the tensor-memory copy: for each expert, K
 *        stage ks (128 bytes of codes along K), 128-row block nb and atom s:
 *        one 512-byte atom holding 128 rows x 4 scales, byte
 *        (n % 32) * 16 + ((n % 128) / 32) * 4 + (scale index % 4), i.e. row
 *        128c + 32j + i sits in 32-bit word 4i + j (the pages' UTCCP row
 *        permutation, _kernel_layout_shard), laid out [E][K stages][NB][S][512]
 *        with NB = round_up(N, 256) / 128 and S = 1 (MXFP8) or 4 (NVFP4)
 *        atoms per stage. Rows past N are zero.
 *   *_gs copied unchanged.
 * Sizes of each kernel-layout tensor: moe_weight_layout_size.
 */
typedef struct moe_weights {
    void*  w13;
    void*  w13_sf;
    float* w13_gs;
    void*  w2;
    void*  w2_sf;
    float* w2_gs;
} moe_weights_t;

#define MOE_W13        0
#define MOE_W13_SF     1
#define MOE_W2         2
#define MOE_W2_SF      3
#define MOE_SHARED_W13     4
#define MOE_SHARED_W13_SF  5
#define MOE_SHARED_W2      6
#define MOE_SHARED_W2_SF   7
#define MOE_W13_GS     8
#define MOE_W2_GS      9

/* Bytes of one kernel-layout tensor (0 where the format has none). Host-only. */
int moe_weight_layout_size(moe_plan_t plan, int32_t which, size_t* bytes);

/*
 * Repack checkpoint-layout routed weights (src, device) into the kernel layout
 * (dst, device, caller-allocated with moe_weight_layout_size bytes each).
 * dst must not alias src. Pure and idempotent (vllm.models.muse_spark.nvidia.
 * mega_moe, finalize_weights; deep_gemm.transform_weights_for_mega_moe).
 */
int moe_transform_weights(moe_plan_t plan, const moe_weights_t* src, moe_weights_t* dst,
                          void* stream);

/* The same for the shared expert (E = 1, I = shared_inter, format = shared_format);
 * the *_gs members are unused. */
int moe_transform_shared_weights(moe_plan_t plan, const moe_weights_t* src, moe_weights_t* dst,
                                 void* stream);

/* ---------------------------------------------------------------- forward */

/*
 * out[t] = bf16( norm( sum_j topk_weights[t,j] * expert_{topk_ids[t,j]}(hidden[t]) + shared(hidden[t]) ) )
 * (DeepGemmMegaMoEExperts.forward; DeepGemmExperts.apply).
 *
 *   num_tokens     T, 0 <= T <= max_tokens (T == 0 launches nothing)
 *   hidden         device bf16 [T, H], row-major
 *   topk_ids       device int32 [T, k]; -1 masks a slot; other ids outside
 *                  [0, E) are treated as masked and set MOE_ERR_BAD_EXPERT_ID
 *   topk_weights   device fp32 [T, k]
 *   weights        routed weights in the kernel layout (moe_transform_weights)
 *   l2_act_scale   device fp32 scalar: NVFP4 L2 input scale (max over experts
 *                  of w2_input_scale, or 1.0); NULL for BF16 / MXFP8
 *   shared         shared expert in the kernel layout, NULL if shared_inter == 0
 *   norm_gamma     device fp32 [H] (applied verbatim), NULL unless post_norm
 *   out            device bf16 [T, H]; must not alias hidden
 *   workspace      device, >= moe_workspace_size(plan, T) bytes
 * Deterministic: the combine sums the k slots in ascending j order in fp32,
 * without atomics.
 */
int moe_forward(moe_plan_t plan, int32_t num_tokens,
                const void* hidden, const int32_t* topk_ids, const float* topk_weights,
                const moe_weights_t* weights, const float* l2_act_scale,
                const moe_weights_t* shared, const float* norm_gamma,
                void* out, void* workspace, size_t workspace_bytes, void* stream);

/*
 * The routed experts on the batched (masked) layout (vllm.model_executor.layers.fused_moe,
 * BatchedDeepGemmExperts.apply: m-grouped GEMMs over [E, max_num_tokens, K] with
 * expert_num_tokens[E], then the activation with requantisation, then the second GEMM).
 *   hidden            bf16 [E, max_tokens, H]: expert e's rows in its own slab
 *   expert_num_tokens int32 [E] (device): the first expert_num_tokens[e] rows of slab e are used
 *   out               bf16 [E, max_tokens, H]: rows m < expert_num_tokens[e] are written, the
 *                     others are left as they are
 * Each used row is quantised in the plan's format (its own NVFP4 scale), then goes through
 * its expert's L1 -> activation -> L2 requantisation -> L2, exactly as a routed row with
 * weight 1. No routing, no combine, no shared expert and no norm (the plan's are ignored).
 * max_tokens: a multiple of 128 (each slab is whole row tiles). Needs the one-kernel GEMM
 * (MOE_FLAG_CTA_PAIR, MOE_FLAG_TILE_128 and MOE_FLAG_SPLIT_GEMM return MOE_ERR_UNSUPPORTED).
 * A count outside [0, max_tokens] is clamped and reported as MOE_ERR_CAPACITY by
 * moe_last_status. Stream-ordered; workspace from moe_batched_workspace_size.
 */
int moe_batched_workspace_size(moe_plan_t plan, int32_t max_tokens, size_t* bytes);
int moe_forward_batched(moe_plan_t plan, int32_t max_tokens, const void* hidden, const int32_t* expert_num_tokens,
                        const moe_weights_t* weights, const float* l2_act_scale, void* out, void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * Synchronise the stream and read (then clear) the device error word of the
 * workspace: *status = MOE_OK, MOE_ERR_BAD_EXPERT_ID or MOE_ERR_TIMEOUT.
 */
int moe_last_status(moe_plan_t plan, void* workspace, void* stream, int32_t* status);

/* ---------------------------------------------------------------- inspection */

#define MOE_REGION_COUNTS     0   /* int32 [E]      tokens routed to each expert */
#define MOE_REGION_OFFSETS    1   /* int32 [E+1]    BLOCK_M-padded segment starts, off[E] = M_pad */
#define MOE_REGION_SRC        2   /* int32 [M_pad]  flat slot t*k+j of each permuted row, -1 = padding */
#define MOE_REGION_INV_PERM   3   /* int32 [T, k]   row of each slot, -1 = masked */
#define MOE_REGION_XQ         4   /* dispatched activations [M_pad_max, H/vpe] (permuted rows) */
#define MOE_REGION_XSF        5   /* their scale atoms [M_pad_max/128][H stages][S][512] */
#define MOE_REGION_XSCALE     6   /* fp32 [T] NVFP4 per-token dispatch scale */
#define MOE_REGION_HQ         7   /* L2 input [M_pad_max, I/vpe] */
#define MOE_REGION_HSF        8   /* its scale atoms */
#define MOE_REGION_H_DEBUG    9   /* fp32 [M_pad_max, I] pre-quantisation h (MOE_FLAG_DEBUG_H) */
#define MOE_REGION_Y         10   /* bf16 [M_pad_max, H] per-row L2 output (alpha applied) */
#define MOE_REGION_META      11   /* int32 [4]: M_pad, number of 128-row tiles, -, - */
#define MOE_REGION_SHARED_Y  12   /* bf16 [T_pad, H] shared-expert output */

/*
 * Offset and size (bytes) of a workspace region for num_tokens tokens, so
 * tests can read the intermediate results of moe_forward. Host-only.
 */
int moe_workspace_region(moe_plan_t plan, int32_t num_tokens, int32_t which,
                         size_t* offset, size_t* bytes);

/* ---------------------------------------------------------------- measurement */

#define MOE_KERNEL_ROUTE      0
#define MOE_KERNEL_DISPATCH   1
#define MOE_KERNEL_L1         2
#define MOE_KERNEL_L2         3
#define MOE_KERNEL_SHARED_L1  4
#define MOE_KERNEL_SHARED_L2  5
#define MOE_KERNEL_COMBINE    6
#define MOE_NUM_KERNELS       7

/*
 * Per-launch timing. With enable = 1 the plan creates CUDA events and every
 * later moe_forward records one before and one after each of its kernel
 * launches on the call's stream (enable = 0 destroys them).
 * moe_plan_kernel_times waits for the last forward's final event and writes
 * the elapsed milliseconds of each launch to ms[MOE_KERNEL_*] (0 for a kernel
 * that did not run); count must be >= MOE_NUM_KERNELS.
 */
int moe_plan_enable_timing(moe_plan_t plan, int32_t enable);
int moe_plan_kernel_times(moe_plan_t plan, float* ms, int32_t count);

/* ---------------------------------------------------------------- permutation without a workspace */

/*
 * The routing permutation of moe_forward (per-expert counts, BLOCK_M = 128
 * padded segment offsets, stable scatter) for callers that must not allocate
 * device memory: a runtime that owns all of HBM through its own pools, or a
 * path where a cudaMalloc is not allowed. The pages have no counterpart of this
 * entry point; it exists for such callers only.
 *
 *   topk_ids        device int32 [T, k], -1 masks a slot (ids outside [-1, E)
 *                   are treated as masked, and no status reports them: the
 *                   kernel's error word stays in the private array)
 *   inv_perm        device int32 [T, k] (output): padded row of each slot, -1 if masked
 *   expert_offsets  device int32 [E + 1] (output): segment starts, [E] = padded total
 * Scratch lives in a fixed device array inside libmoe.so (about 1.06 MB per
 * GPU, held until the process exits): T * k + E * 127 must be <= 262144
 * (else MOE_ERR_CAPACITY, nothing launched); 1 <= k <= 32, 1 <= E <= 512.
 * The first call on a device sets that device up (looks up the array's
 * address); make it before any stream capture. That set-up belongs to the
 * CUDA context it was made in: do not call this again after a
 * cudaDeviceReset in the same process. Calls share the array: calls whose GPU
 * work overlaps race. Allocates nothing.
 */
int moe_permute_noalloc(const int32_t* topk_ids, int32_t num_tokens, int32_t top_k, int32_t num_experts,
                        int32_t* inv_perm, int32_t* expert_offsets, void* stream);

/*
 * Limit of each bounded wait inside the GEMM kernels (default 2 s; 0 restores
 * the default). A wait that runs out makes the kernel record MOE_ERR_TIMEOUT,
 * wait for its own copies and MMAs, free its tensor memory and return, leaving
 * the CUDA context usable; moe_last_status reports it. Used to test that path.
 */
int moe_plan_set_wait_timeout(moe_plan_t plan, uint64_t timeout_ns);

/* Static string for a status code. */
const char* moe_error_string(int32_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
