// moe_internal.h -- pool layout and kernel launchers shared inside libmoe.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cstdlib>
#include <cuda_runtime.h>

#include "moe.h"

namespace moe {

constexpr int kGroup = 128;       // quantization group (elements)
constexpr int kTileTokens = 32;   // tokens per placement tile (one mask word)
constexpr int kMidTileTokens = 16;      // tile of the three-launch plan for mid-size batches
constexpr int kMidTileMaxTokens = 2048; // largest batch that takes it

// Lanes per token in the three-launch route kernel: the fewest of 8, 16, 32
// that keep at most 8 keys a lane and leave a lane per (token, j) for the
// gates.
inline int route_lanes(int E, int k) {
    const int kp = k <= 1 ? 1 : 1 << (32 - __builtin_clz((unsigned)(k - 1)));
    return (E <= 64 && kp <= 8) ? 8 : (E <= 128 && kp <= 16) ? 16 : 32;
}

// Tokens per tile of the three-launch plan: 16 for batches of 513 to 2048
// tokens whose tokens take a whole warp (512-thread CTAs, so that fewer
// warps route at once on an SM), else 32.  Batches of up to 512 tokens take
// it only when the cluster plan is refused.
inline int route_tile_tokens(int T, int E, int k) {
    return (T > 512 && T <= kMidTileMaxTokens && route_lanes(E, k) == 32) ? kMidTileTokens : kTileTokens;
}

// Tile-count scratch of a plan of T tokens: ceil(T / tile tokens) columns.
inline int route_tiles(int T, int E, int k) {
    const int tt = route_tile_tokens(T, E, k);
    return (T + tt - 1) / tt;
}
constexpr int kMaxSets = 4;

// Byte offsets (from the workspace base) of one buffer set's regions.
struct SetLayout {
    size_t codes, scales, ex_out;
    size_t topk_e, phys, gates, slot, src_token, src_k, counts, offsets;
    size_t tile_hist, local_rank;
    size_t x_stage, logits_stage, y_stage;
};

struct Geometry {
    moe_desc d;
    int64_t rows;        // T_max * k
    int32_t G;           // H / 128
    int32_t Gs;          // G rounded up to a multiple of 4 (16-byte scale rows)
    int32_t tiles_max;   // the most tile columns any T <= T_max uses (route_tiles)
    size_t error_word;   // offset of the shared device error word
    size_t ticket;       // offset of n_sets int32 plan tickets (single-launch plan)
    size_t control_bytes;// error word + tickets, zeroed by moe_pool_clear_error
    SetLayout set[kMaxSets];
    size_t total;
};

int make_geometry(const moe_desc* d, Geometry* g);

// Launch with programmatic stream serialization, so that the kernel can be
// scheduled while the previous kernel in the stream drains (the kernel itself
// waits for it in grid_dependency_sync before touching global memory).
// `priority` != 0 adds a launch priority (cudaLaunchAttributePriority; lower
// numbers are more urgent).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_at(int priority, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributePriority;
    attr[1].val.priority = priority;
    cfg.attrs = attr;
    cfg.numAttrs = priority != 0 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// As launch_pdl_at, with the grid launched as thread-block clusters of
// `cluster_x` CTAs (cudaLaunchAttributeClusterDimension).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(int priority, unsigned cluster_x, void (*kernel)(KArgs...), dim3 grid, dim3 block,
                               size_t smem, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[3];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    attr[2].id = cudaLaunchAttributePriority;
    attr[2].val.priority = priority;
    cfg.attrs = attr;
    cfg.numAttrs = priority != 0 ? 3 : 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
    return launch_pdl_at(0, kernel, grid, block, smem, s, args...);
}

// Whether the current device launches thread-block clusters (looked up once).
inline bool cluster_launch_supported() {
    static const bool v = [] {
        // MOE_PLAN_NO_CLUSTER=1 takes the ticket plan instead (a device or a
        // partition that refuses clusters takes it anyway, per launch).
        const char* off = std::getenv("MOE_PLAN_NO_CLUSTER");
        if (off != nullptr && off[0] == '1' && off[1] == '\0') return false;
        int dev = 0, ok = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&ok, cudaDevAttrClusterLaunch, dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return false;
        }
        return ok != 0;
    }();
    return v;
}

// The most urgent launch priority the device offers (cudaDeviceGetStreamPriorityRange's
// "greatest" value; 0 where the device has no priorities).  Looked up once.
inline int most_urgent_priority() {
    static const int v = [] {
        int least = 0, greatest = 0;
        if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        return greatest;
    }();
    return v;
}

// Launchers: enqueue on `s`, return cudaGetLastError() after the launch(es).
// Each adds the number of kernels it launched to *launches.
cudaError_t launch_plan(const float* logits, int T, int E, int P, int k,
                        const int32_t* rep_off, const int32_t* rep_ids,
                        int32_t* topk_e, float* gates, int32_t* phys,
                        int32_t* tile_hist, int32_t* local_rank,
                        int32_t* counts, int32_t* offsets, int32_t* slot,
                        int32_t* src_token, int32_t* src_k, int32_t* err,
                        int32_t* ticket /* zeroed int32, or NULL: always three launches */,
                        cudaStream_t s, uint64_t* launches);

// x_early: read x before waiting for the preceding kernel (see moe_dispatch_after_plan).
cudaError_t launch_dispatch(const uint16_t* x, int T, int H, int k, const int32_t* slot,
                            int8_t* codes, float* scales, int Gs, int32_t* err, bool x_early,
                            cudaStream_t s, uint64_t* launches);

cudaError_t launch_identity_experts(const int8_t* codes, const float* scales, int rows, int H, int Gs,
                                    uint16_t* ex_out, cudaStream_t s, uint64_t* launches);

cudaError_t launch_combine(const uint16_t* ex_out, const int32_t* slot, const float* gates,
                           int T, int H, int k, uint16_t* y, int32_t* err,
                           cudaStream_t s, uint64_t* launches);

}  // namespace moe

struct moe_pool {
    moe::Geometry geo;
    char* base;                       // device workspace
    int32_t planned_T[moe::kMaxSets]; // T of the last moe_plan per set (-1 = none)
    uint64_t launches;
};
