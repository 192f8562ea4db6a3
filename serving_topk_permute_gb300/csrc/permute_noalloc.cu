// permute_noalloc.cu -- the routing permutation for callers that must not allocate
// device memory.
//
// Some callers cannot hand the library a workspace: a serving runtime that
// reserves all of HBM up front for its own pools (weights, KV cache) and owns
// every byte through its allocator, or a latency-critical path where a
// cudaMalloc (and the device synchronisation it can imply) is not allowed.
// moe_permute_noalloc runs the same routing kernel as moe_forward, but keeps
// the kernel's scratch (per-expert counts, the padded row -> slot map, the
// row-tile map, the meta words and the error word) in one file-scope device
// array of fixed size instead of a caller workspace.
//
// Properties a caller must know:
//   - Scratch capacity: NOALLOC_MAX_ROWS padded rows, i.e. calls with
//     num_tokens * top_k + num_experts * 127 > 262144 are rejected with
//     MOE_ERR_CAPACITY before anything is launched.
//   - Every GPU that loads libmoe.so holds the array (about 1.06 MB) until the
//     process exits.
//   - The first call on a device does the set-up for that device: it looks up
//     the array's device address (cudaGetSymbolAddress) and sets the routing
//     kernel's shared-memory limit. Make that first call before any stream
//     capture.
//   - All calls share the one array and it keeps the previous call's contents:
//     calls whose GPU work overlaps (different streams without ordering
//     between them) race on it. The kernel itself clears what must start at
//     zero (the error word) and writes every other word before reading it.
//   - Ids outside [-1, E) are treated as masked. The kernel's error word stays
//     in the private array and no call reads it back, so such ids produce no
//     status; moe_forward reports them through moe_last_status.
//   - The cached set-up belongs to the CUDA context it was made in: after a
//     cudaDeviceReset the array's address and the kernel attribute are stale,
//     so the entry point must not be used again in that process.
//   - Nothing here allocates: no cudaMalloc, no cudaFree, no allocating
//     library routine.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace {

constexpr int64_t NOALLOC_MAX_ROWS = 1 << 18;            // 262144 padded permuted rows
constexpr int NOALLOC_MAX_EXPERTS = 512;
constexpr int64_t OFF_ERR = 0;                           // [16]   error word (+ padding)
constexpr int64_t OFF_META = 16;                         // [16]   M_pad, row tiles
constexpr int64_t OFF_CNT = 32;                          // [512]  tokens per expert
constexpr int64_t OFF_TILES = OFF_CNT + NOALLOC_MAX_EXPERTS;                      // [2048] row tile -> expert
constexpr int64_t OFF_SRC = OFF_TILES + NOALLOC_MAX_ROWS / moe::BM;              // [262144] row -> slot
constexpr int64_t NOALLOC_INTS = OFF_SRC + NOALLOC_MAX_ROWS;

static __device__ __align__(256) int g_noalloc_route_scratch[NOALLOC_INTS];

constexpr int MAX_DEVICES = 64;
std::mutex g_setup_mutex;
int* g_scratch_ptr[MAX_DEVICES] = {};  // device address of the array, per device (set-up done when non-null)

// once per device, with that device current
int setup_device(int dev, int** out) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_route_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        if (moe::route_prepare(NOALLOC_MAX_EXPERTS) != cudaSuccess) return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<int*>(p);
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" int moe_permute_noalloc(const int32_t* topk_ids, int32_t num_tokens, int32_t top_k, int32_t num_experts,
                                   int32_t* inv_perm, int32_t* expert_offsets, void* stream) {
    if (num_tokens < 0 || top_k < 1 || top_k > 32 || num_experts < 1 || num_experts > NOALLOC_MAX_EXPERTS)
        return MOE_ERR_INVALID_ARG;
    if (!expert_offsets || (num_tokens > 0 && (!topk_ids || !inv_perm))) return MOE_ERR_INVALID_ARG;
    const int64_t R = (int64_t)num_tokens * top_k;
    if (R + (int64_t)num_experts * (moe::BM - 1) > NOALLOC_MAX_ROWS) return MOE_ERR_CAPACITY;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return MOE_ERR_CUDA;
    int* s = nullptr;
    const int rc = setup_device(dev, &s);
    if (rc != MOE_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the routing kernel zeroes the error word and writes every other word it reads first
    if (moe::launch_route(topk_ids, num_tokens, top_k, num_experts, moe::BM, s + OFF_CNT, expert_offsets, s + OFF_SRC,
                          inv_perm, s + OFF_TILES, s + OFF_META, s + OFF_ERR, st) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
