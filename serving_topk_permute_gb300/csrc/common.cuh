// common.cuh -- shared device helpers for the sm_103a MoE kernels: inline PTX for
// mbarriers (bounded waits), TMA / bulk copies, tcgen05 (tensor memory, MMA,
// scale-factor copies, loads), FP8 / FP4 conversions, and the layout formulas
// every kernel agrees on.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

namespace moe {

// ------------------------------------------------------------------ tile geometry
constexpr int BM = 128;            // rows per MMA tile (= BLOCK_M of the routing)
constexpr int BN_MAX = 256;        // widest MMA tile (weight rows); tiles are 128 or 256 wide
constexpr int NBLK = 128;          // weight rows per scale-atom block and per gate/up interleave unit
constexpr int BK_BYTES = 128;      // bytes of codes per K stage (one 128-byte swizzle row)
constexpr int A_BOX_ROWS = 32;     // the one-kernel GEMM loads a row tile's used rows in boxes this high
constexpr int ATOM_BYTES = 512;    // one scale-factor atom: 128 rows x 4 scales
constexpr int EPI_WARPS = 16;      // 4 per tensor-memory lane quarter, each on a quarter of the columns
constexpr int GEMM_THREADS = 64 + 32 * EPI_WARPS;  // warp 0 TMA producer, warp 1 MMA issuer, then epilogue
constexpr int TMEM_COLS = 512;
// limit of the end-of-kernel waits for a CTA's own copies and MMAs, independent of the
// (configurable) limit of the pipeline waits, so a CTA that gave up never exits with
// work in flight
constexpr unsigned long long DRAIN_TIMEOUT_NS = 2000000000ull;

// per-format constants
__host__ __device__ constexpr int fmt_elem_bits(int fmt) { return fmt == MOE_FMT_BF16 ? 16 : (fmt == MOE_FMT_MXFP8 ? 8 : 4); }
// scale-factor atoms per K stage (each atom covers 4 scale blocks along K): a 128-byte
// stage holds 128 MXFP8 (4 blocks of 32), 256 NVFP4 (16 blocks of 16) or 256 MXFP4
// (8 blocks of 32) elements
__host__ __device__ constexpr int fmt_sf_atoms(int fmt) {
    return fmt == MOE_FMT_BF16 ? 0 : (fmt == MOE_FMT_MXFP8 ? 1 : (fmt == MOE_FMT_MXFP4 ? 2 : 4));
}
// elements per scale block
__host__ __device__ constexpr int fmt_sf_block(int fmt) { return fmt == MOE_FMT_NVFP4 ? 16 : 32; }
// bytes of one row of K elements
__host__ __device__ inline int64_t fmt_row_bytes(int fmt, int64_t K) { return K * fmt_elem_bits(fmt) / 8; }
// number of 128-byte K stages for K elements
__host__ __device__ inline int64_t fmt_k_stages(int fmt, int64_t K) { return fmt_row_bytes(fmt, K) / BK_BYTES; }

// The routing kernel splits the flat slots s = t*k + j into ROUTE_WARPS contiguous
// chunks, one per warp; a slot's rank inside its expert is the chunk's base for the
// expert plus the number of equal ids before it in the chunk.
constexpr int ROUTE_WARPS = 32;
__host__ __device__ inline int route_chunk(int64_t R) { return (int)(((R + ROUTE_WARPS - 1) / ROUTE_WARPS + 31) / 32 * 32); }

// Byte offset of scale block kb of row r in an activation scale-atom array laid
// out [row tile][K stage][S atoms][512]: within an atom, row m = 32j + i and
// scale b (of 4) sit at byte 16i + 4j + b.
__host__ __device__ inline int64_t act_sf_offset(int64_t r, int64_t kb, int S, int64_t nks) {
    const int64_t mt = r / BM, m = r % BM;
    const int64_t ks = kb / (4 * S), s = (kb / 4) % S, b = kb % 4;
    return ((mt * nks + ks) * S + s) * ATOM_BYTES + (m % 32) * 16 + (m / 32) * 4 + b;
}

// Weight scale atoms are laid out [E][K stage][N blocks][S atoms][512] with 128-row
// blocks and N blocks = round_up(N, 256) / 128 (rows past N are zero), so the atoms of
// one K stage of any 128- or 256-row tile are one contiguous run.
__host__ __device__ inline int64_t wt_sf_blocks(int64_t N) { return (N + BN_MAX - 1) / BN_MAX * (BN_MAX / NBLK); }

// w13 gate/up interleave: kernel row 128 b + 64 h + r (h 0 = gate, 1 = up, r < 64)
// holds checkpoint row h * I + 64 b + r.
__host__ __device__ inline int64_t w13_src_row(int64_t n, int64_t I) {
    const int64_t b = n / NBLK, h = (n % NBLK) / 64, r = n % 64;
    return h * I + b * 64 + r;
}

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ inline int64_t align_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// ------------------------------------------------------------------ device error word
__device__ inline void set_error(int* err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// Programmatic dependent launch. A kernel launched with the programmatic-serialisation
// attribute may start while its predecessor in the stream is still running: it does
// its set-up (shared memory, barriers, tensor memory), then grid_dep_wait() blocks
// until the predecessor grid has completed and its writes are visible. Every global
// read or write of the forward's buffers comes after that wait. grid_dep_launch()
// then lets the successor start its own set-up. A kernel launched without the
// attribute returns from both at once.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ------------------------------------------------------------------ cross-CTA flags in global memory
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_gpu_add(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// orders this thread's generic-proxy global accesses with its later (or earlier)
// async-proxy ones (TMA): data written with st.global and read back by TMA
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ shared memory / mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// one bounded test of a barrier phase: the thread may suspend for at most hint_ns
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// a non-suspending test of a barrier phase
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// limits below this are polled without suspending (a suspended try_wait may sleep longer)
constexpr uint64_t SHORT_WAIT_NS = 1000000ull;

// the longest single suspension inside a bounded wait
__device__ __forceinline__ uint32_t wait_hint(uint64_t timeout_ns) {
    return (uint32_t)(timeout_ns < 1000000ull ? timeout_ns : 1000000ull);
}

// Wait for the phase of `bar` with parity `parity` to complete, giving up after
// timeout_ns (or as soon as *abort is set). Returns false on give-up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                          const volatile int* abort) {
    const uint32_t hint = wait_hint(timeout_ns);
    if (timeout_ns < SHORT_WAIT_NS) {
        for (uint64_t i = 0; i < 32 * (1 + timeout_ns / 256); ++i)
            if (mbar_test_wait(bar, parity)) return true;
        return false;
    }
    if (mbar_try_wait(bar, parity, hint)) return true;
    const uint64_t t0 = globaltimer_ns();
    // rounds of 32 polls: bounds the wait even where the global timer ticks coarsely
    const uint64_t max_rounds = 1 + timeout_ns / 256;
    for (uint64_t round = 0;; ++round) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity, hint)) return true;
        if (*abort) return false;
        if (round >= max_rounds || globaltimer_ns() - t0 > timeout_ns) return false;
    }
}

// Wait until *flag >= target (read with acquire at GPU scope), giving up after
// timeout_ns or as soon as *abort is set. Returns false on give-up.
__device__ __forceinline__ bool flag_wait_geq(const uint32_t* flag, uint32_t target, uint64_t timeout_ns,
                                              const volatile int* abort) {
    if (ld_acquire_gpu(flag) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    const uint64_t max_rounds = 1 + timeout_ns / 64;  // bounds the wait even where the timer ticks coarsely
    for (uint64_t round = 0;; ++round) {
        __nanosleep(64);
        if (ld_acquire_gpu(flag) >= target) return true;
        if (*abort) return false;
        if (round >= max_rounds || globaltimer_ns() - t0 > timeout_ns) return false;
    }
}

// ------------------------------------------------------------------ TMA / bulk copies (global -> shared)
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// Tiled loads of one CTA of a CTA pair (cta_group::2): the data lands in the issuing
// CTA's shared memory at dst, and the completed bytes are counted on the barrier at
// bar_cl, a shared::cluster address that may be in either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_cg2(uint32_t dst, const CUtensorMap* map, uint32_t bar_cl, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cl), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d_cg2(uint32_t dst, const CUtensorMap* map, uint32_t bar_cl, int x, int y,
                                                int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cl), "r"(x), "r"(y), "r"(z)
        : "memory");
}

// The same 3-D tiled load with an L2 cache policy (from make_policy_*): weights that one
// row tile streams once are marked evict-first, weights that many row tiles reuse evict-last.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                 int z, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "l"(policy)
        : "memory");
}
__device__ __forceinline__ uint64_t make_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t make_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// prefetch one tensor tile into L2 (no shared memory, no barrier)
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// plain bulk copy: both addresses 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// arrive on `bar` once every tcgen05 operation issued so far by this thread has completed
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start >> 4 in bits 0-13,
// leading byte offset >> 4 in 16-29, stride byte offset >> 4 in 32-45, the
// fixed 0b001 in 46-48, swizzle mode in 61-63 (2 = 128-byte swizzle, 0 = none).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)(swizzle & 7) << 61;
    return d;
}

// K-major operand tile whose rows are 128 bytes, 128-byte swizzled (as TMA
// writes it): 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t kmajor_sw128_desc(uint32_t saddr) { return smem_desc(saddr, 16, 1024, 2); }

// 32 rows x 16 bytes, no swizzle (the source of a 32x128b tensor-memory copy)
__device__ __forceinline__ uint64_t sf_atom_desc(uint32_t saddr) { return smem_desc(saddr, 0, 128, 0); }

// copy one scale-factor atom (32 lanes x 128 bits, replicated to the four lane quarters)
__device__ __forceinline__ void tc_cp_sf_atom(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}

// Instruction descriptors (M = 128, N = n, both operands K-major).
// kind::f16: D fp32 (bits 4-5 = 1), A/B bf16 (bits 7-9, 10-12 = 1), N>>3 at 17, M>>4 at 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}
// kind::mxf8f6f4: A/B E4M3 (0), scale type UE8M0 (bit 23), scale ids: B at 4-5, A at 29-30.
__host__ __device__ constexpr uint32_t idesc_mxf8(int n, uint32_t sf_id) {
    return (sf_id << 4) | ((uint32_t)(n >> 3) << 17) | (1u << 23) | ((uint32_t)(BM >> 4) << 24) | (sf_id << 29);
}
// kind::mxf4nvf4: A/B E2M1 (1), scale type UE4M3 (bit 23 = 0).
__host__ __device__ constexpr uint32_t idesc_nvf4(int n) {
    return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);
}
// kind::mxf4nvf4 with scale_vec::2X (MXFP4): A/B E2M1, scale type UE8M0 (bit 23); each
// MMA (K = 64) takes two scales per row, bytes sf_id and sf_id + 1 (sf_id 0 or 2) of
// the row's 32-bit scale column.
__host__ __device__ constexpr uint32_t idesc_mxf4(int n, uint32_t sf_id) {
    return (sf_id << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | (1u << 23) |
           ((uint32_t)(BM >> 4) << 24) | (sf_id << 29);
}

// load 32 consecutive fp32 columns of this warp's 32 lanes (one row per thread)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// four consecutive 32-bit columns of the 32 tensor-memory lanes of this warp's quarter:
// lane i of the warp writes v to lane i of the quarter (taddr carries the quarter's first lane)
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint4& v) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ clusters and 2-CTA (cta_group::2) MMA
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// all threads of all CTAs of the cluster
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// the shared::cluster address of the same shared variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// Arrive on a barrier of another CTA of the cluster. Default (release, CTA scope)
// semantics: the callers publish no writes of their own (the data they signal was
// written by TMA and observed through a barrier, or read from tensor memory and
// ordered by tcgen05.fence). A cluster-scope release measured ~1300 cycles per
// arrive on GB300, which throttled a one-arrive-per-stage pipeline to half speed.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// the same with an expected transaction count (bytes that copies will complete on it)
__device__ __forceinline__ void mbar_arrive_expect_tx_cluster(uint32_t cluster_addr, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_addr), "r"(bytes)
                 : "memory");
}
// arrive with cluster-scope release: the caller's earlier shared::cluster stores are
// visible to a thread that observes the phase with an acquire.cluster wait
__device__ __forceinline__ void mbar_arrive_release_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cl(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_test_wait_cl(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// as mbar_wait, with cluster-scope acquire (arrivals from the peer CTA)
__device__ __forceinline__ bool mbar_wait_cl(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                             const volatile int* abort) {
    const uint32_t hint = wait_hint(timeout_ns);
    if (timeout_ns < SHORT_WAIT_NS) {
        for (uint64_t i = 0; i < 32 * (1 + timeout_ns / 256); ++i)
            if (mbar_test_wait_cl(bar, parity)) return true;
        return false;
    }
    if (mbar_try_wait_cl(bar, parity, hint)) return true;
    const uint64_t t0 = globaltimer_ns();
    // rounds of 32 polls: bounds the wait even where the global timer ticks coarsely
    const uint64_t max_rounds = 1 + timeout_ns / 256;
    for (uint64_t round = 0;; ++round) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait_cl(bar, parity, hint)) return true;
        if (*abort) return false;
        if (round >= max_rounds || globaltimer_ns() - t0 > timeout_ns) return false;
    }
}
// tensor memory of a CTA pair: issued by one warp in each of the two CTAs
__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// arrive on the barrier at this shared offset in every CTA of cta_mask once the issued tcgen05 work completes
__device__ __forceinline__ void tc_commit2_mc(uint32_t bar, uint16_t cta_mask) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                     bar),
                 "h"(cta_mask)
                 : "memory");
}
// copy one scale atom from each CTA's shared memory into its own tensor memory
__device__ __forceinline__ void tc_cp2_sf_atom(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
__device__ __forceinline__ void mma2_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma2_mxf8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma2_mxf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma2_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
        : "memory");
}
// instruction descriptors with an explicit M (128 for one CTA, 256 for a CTA pair)
__host__ __device__ constexpr uint32_t idesc_m(uint32_t idesc, int m) {
    return (idesc & ~(0x1Fu << 24)) | ((uint32_t)(m >> 4) << 24);
}

// ------------------------------------------------------------------ conversions
// two fp32 -> packed E4M3 pair, round to nearest even, saturate to +-448; `lo` goes to the low byte
__device__ __forceinline__ uint16_t cvt_e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
// two fp32 -> packed E2M1 pair, round to nearest even, saturate to +-6; `lo` goes to the low nibble
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r;
}
// one E4M3 byte -> fp32 (exact)
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
    uint32_t h2;
    const uint16_t in = (uint16_t)((byte & 0xFF) | ((byte & 0xFF) << 8));  // same code in both halves
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFF)));
}

// UE8M0 exponent of a block: the smallest e with amax <= 448 * 2^e (0 for amax == 0),
// decided exactly from frexp: amax = f * 2^p, f in [0.5, 1), 448 = 0.875 * 2^9.
__device__ __forceinline__ int ue8m0_exponent(float amax) {
    if (!(amax > 0.0f)) return 0;
    int p;
    const float f = frexpf(amax, &p);
    int e = (f <= 0.875f) ? p - 9 : p - 8;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}
// MXFP4 block exponent: the smallest e with amax <= 6 * 2^e. With amax = f * 2^p,
// f in [0.5, 1): 6 * 2^(p-3) = 0.75 * 2^p, so e = p - 3 when f <= 0.75, else p - 2.
__device__ __forceinline__ int ue8m0_exponent_fp4(float amax) {
    if (!(amax > 0.0f)) return 0;
    int p;
    const float f = frexpf(amax, &p);
    int e = (f <= 0.75f) ? p - 3 : p - 2;
    return e < -127 ? -127 : (e > 127 ? 127 : e);
}

}  // namespace moe
