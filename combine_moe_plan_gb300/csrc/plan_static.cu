// plan_static.cu -- moe_plan_static: the routing-metadata pass for callers
// that cannot allocate device memory.
//
// moe_plan keeps its scratch (per-tile expert counts and in-tile ranks) in the
// pool workspace the caller allocated.  Some callers have no allocator at
// all: code running inside a CUDA graph that was built elsewhere, plugins
// whose host framework owns every device allocation, or processes that must
// not grow their device footprint after start-up.  They pass only their own
// inputs and outputs; the scratch lives in the fixed-size array below, which
// is part of this library's device image.
//
// Costs and limits of that choice:
//   - kStaticScratchBytes (4 MiB) of device memory is held on every GPU that
//     loads this library's device code, until the process exits.
//   - Every call shares the one array, so calls whose kernels overlap on the
//     GPU (different streams, or different host threads) race on it and give
//     wrong slots.  Serialize them, e.g. issue them on one stream.
//   - Nothing in the array has to start at zero: the route kernel writes every
//     entry the later kernels of the same call read, so leftovers from an
//     earlier call are never seen.
//   - The first call on each device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current and caches it; make that
//     first call before any stream capture begins.
#include <mutex>

#include "moe_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_plan_scratch[kStaticScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_plan_scratch on the current device (looked up once per
// device).  Host code only ever sees a host-side stand-in for the array's
// name, so the address must come from the runtime.
int static_scratch(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_SIZE;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return MOE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

}  // namespace

extern "C" MOE_API int moe_plan_static(const float* logits, int32_t T, int32_t E, int32_t P, int32_t k,
                                       const int32_t* rep_off, const int32_t* rep_ids, int32_t* topk_e,
                                       float* gates, int32_t* phys, int32_t* counts, int32_t* offsets,
                                       int32_t* slot, int32_t* src_token, int32_t* src_k, int32_t* error_word,
                                       void* stream) {
    if (T == 0) {  // an empty batch: every expert window is empty
        if (counts == nullptr || offsets == nullptr) return MOE_ERR_NULL;
        if (P < 1 || P > 4096) return MOE_ERR_SIZE;
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        if (cudaMemsetAsync(counts, 0, (size_t)P * sizeof(int32_t), s) != cudaSuccess ||
            cudaMemsetAsync(offsets, 0, (size_t)(P + 1) * sizeof(int32_t), s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    if (logits == nullptr || topk_e == nullptr || gates == nullptr || phys == nullptr || counts == nullptr ||
        offsets == nullptr || slot == nullptr || src_token == nullptr || src_k == nullptr ||
        error_word == nullptr)
        return MOE_ERR_NULL;
    if ((rep_off == nullptr) != (rep_ids == nullptr)) return MOE_ERR_NULL;
    if (T < 1 || T > (1 << 20) || E < 1 || E > 1024 || P < E || P > 4096 || k < 1 || k > E || k > 32)
        return MOE_ERR_SIZE;
    if (rep_off == nullptr && P != E) return MOE_ERR_REPLICA;
    const void* ptrs[] = {logits, topk_e, gates, phys, counts, offsets, slot, src_token, src_k, error_word};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MOE_ERR_ALIGN;
    if (rep_off != nullptr && (!aligned16(rep_off) || !aligned16(rep_ids))) return MOE_ERR_ALIGN;

    const size_t n_tiles = ((size_t)T + moe::kTileTokens - 1) / moe::kTileTokens;
    const size_t hist_bytes = round256((size_t)P * n_tiles * sizeof(int32_t));
    const size_t rank_bytes = round256((size_t)T * (size_t)k * sizeof(int32_t));
    if (hist_bytes + rank_bytes > kStaticScratchBytes) return MOE_ERR_SIZE;

    void* base = nullptr;
    int rc = static_scratch(&base);
    if (rc != MOE_OK) return rc;
    int32_t* tile_hist = static_cast<int32_t*>(base);
    int32_t* local_rank = reinterpret_cast<int32_t*>(static_cast<char*>(base) + hist_bytes);
    uint64_t launches = 0;
    cudaError_t e = moe::launch_plan(logits, T, E, P, k, rep_off, rep_ids, topk_e, gates, phys, tile_hist,
                                     local_rank, counts, offsets, slot, src_token, src_k, error_word, nullptr,
                                     static_cast<cudaStream_t>(stream), &launches);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
