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
//     (cudaGetSymbolAddress) with that device current and caches it, keyed
//     by the device and by the unique id of its current context: a context
//     destroyed and re-created (cudaDeviceReset) loads the module again,
//     possibly at another address, and its new id makes the next call look
//     the address up again.  Make the first call on a device before any
//     stream capture begins.
#include <cuda.h>  // CUcontext / CUresult types only: the two driver calls are looked up at run time

#include <mutex>

#include "moe_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_plan_scratch[kStaticScratchBytes];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

struct ScratchCache {
    bool valid = false;
    unsigned long long ctx_id = 0;
    void* addr = nullptr;
};

std::mutex g_scratch_mu;
ScratchCache g_scratch[kMaxDevices];
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// The unique id of the calling thread's current context, through driver entry
// points the runtime hands out (no driver library is linked).  Caller holds
// g_scratch_mu.
int current_context_id(unsigned long long* id) {
    if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr) {
        void* f1 = nullptr;
        void* f2 = nullptr;
        cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound;
        cudaDriverEntryPointQueryResult q2 = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) !=
                cudaSuccess ||
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
            q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || f1 == nullptr ||
            f2 == nullptr)
            return MOE_ERR_CUDA;
        g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
        g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f2);
    }
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return MOE_ERR_CUDA;
    return g_ctx_get_id(ctx, id) == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// Device address of g_plan_scratch on the current device.  Host code only
// ever sees a host-side stand-in for the array's name, so the address must
// come from the runtime; it is looked up once per device and context.
int static_scratch(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_SIZE;
    // Makes the device's primary context current in this thread (re-creating
    // it after a reset), so that the id below is that of the context the
    // kernels will run in.
    if (cudaSetDevice(dev) != cudaSuccess) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    unsigned long long id = 0;
    const int rc = current_context_id(&id);
    if (rc != MOE_OK) return rc;
    ScratchCache& c = g_scratch[dev];
    if (!c.valid || c.ctx_id != id) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_plan_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
        c.addr = p;
        c.ctx_id = id;
        c.valid = true;
    }
    *out = c.addr;
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
    // The same checks for every T; only logits may be NULL for an empty batch.
    if ((logits == nullptr && T != 0) || topk_e == nullptr || gates == nullptr || phys == nullptr ||
        counts == nullptr || offsets == nullptr || slot == nullptr || src_token == nullptr || src_k == nullptr ||
        error_word == nullptr)
        return MOE_ERR_NULL;
    if ((rep_off == nullptr) != (rep_ids == nullptr)) return MOE_ERR_NULL;
    if (T < 0 || T > (1 << 20) || E < 1 || E > 1024 || P < E || P > 4096 || k < 1 || k > E || k > 32)
        return MOE_ERR_SIZE;
    if (rep_off == nullptr && P != E) return MOE_ERR_REPLICA;
    const void* ptrs[] = {logits, topk_e, gates, phys, counts, offsets, slot, src_token, src_k, error_word};
    for (const void* p : ptrs)
        if (!aligned16(p)) return MOE_ERR_ALIGN;
    if (rep_off != nullptr && (!aligned16(rep_off) || !aligned16(rep_ids))) return MOE_ERR_ALIGN;

    const size_t n_tiles = (size_t)moe::route_tiles(T, E, k);
    const size_t hist_bytes = round256((size_t)P * n_tiles * sizeof(int32_t));
    const size_t rank_bytes = round256((size_t)T * (size_t)k * sizeof(int32_t));
    if (hist_bytes + rank_bytes > kStaticScratchBytes) return MOE_ERR_SIZE;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (T == 0) {  // an empty batch: every expert window is empty
        if (cudaMemsetAsync(counts, 0, (size_t)P * sizeof(int32_t), s) != cudaSuccess ||
            cudaMemsetAsync(offsets, 0, (size_t)(P + 1) * sizeof(int32_t), s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }

    void* base = nullptr;
    const int rc = static_scratch(&base);
    if (rc != MOE_OK) return rc;
    int32_t* tile_hist = static_cast<int32_t*>(base);
    int32_t* local_rank = reinterpret_cast<int32_t*>(static_cast<char*>(base) + hist_bytes);
    uint64_t launches = 0;
    cudaError_t e = moe::launch_plan(logits, T, E, P, k, rep_off, rep_ids, topk_e, gates, phys, tile_hist,
                                     local_rank, counts, offsets, slot, src_token, src_k, error_word, nullptr, s,
                                     &launches);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
