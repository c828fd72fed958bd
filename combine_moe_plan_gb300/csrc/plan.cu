// plan.cu -- routing metadata for FusedDispatch: top-k, gates, replica pick,
// per-expert histogram, exclusive scan and stable slot assignment.
//
// CloudMatrix384 write-up: "FusedDispatch and FusedCombine" (routing metadata
// is the first of the three exchanges the fused operators absorb), "Decode
// Phase" (redundant experts for load balancing), "Prefill Phase" (metadata
// generation and token reordering before dispatch).  StrataCL analysis,
// section 3.5: token placement -> expert-window aggregation.
//
// The per-tile routing body (route_tile) is in route.cuh.  Three launches for
// large batches (one for small ones: plan_cluster_kernel, plan_single_kernel):
//   route_tile   one CTA of 32 warps per tile of 32 tokens, one warp per
//                token: k rounds of warp arg-max by redux.sync over each
//                lane's cached two largest keys (ties -> lower expert id).
//                The CTA then computes the gates (the softmax over the k
//                selected logits, rounded once to fp32: from float pairs, see
//                dword.cuh, with fp64 for the rare token the pairs cannot
//                settle), applies the replica map, and sets
//                bit t of a shared-memory mask per physical expert.  From the
//                mask: the tile's count per expert (popc) and each copy's rank
//                among earlier tokens of the tile (popc of the lower bits).
//   column_scan  one warp per physical expert: exclusive scan of the tile
//                counts down the tiles -> per-tile base inside the expert's
//                window; the column total is counts[p].
//   assign       every CTA scans counts[] in shared memory (offsets); each
//                thread places one (t, j): slot = offsets[p] + tile base +
//                in-tile rank, and writes the inverse map.
// No atomics decide any position, so the result is deterministic and equal
// to a stable counting sort by (expert, token).
#include <cfloat>
#include <climits>

#include "dword.cuh"
#include "moe_internal.h"
#include "ptx.cuh"
#include "trace.cuh"

MOE_TRACE_BUFFERS(tr_route)
MOE_TRACE_BUFFERS(tr_single)
MOE_TRACE_BUFFERS(tr_scan)
MOE_TRACE_BUFFERS(tr_assign)

#include "route.cuh"  // route_tile and its helpers (uses tr_route, tr_single)

namespace moe {
namespace {

// Batches of at most this many 32-token tiles that do not take the cluster
// plan (clusters refused) are planned in one launch, the ticket kernel.  Its
// single-CTA tail grows with the batch: as a graph it ties the three launches
// at 3 tiles and loses at 8 and more (256 tokens 14.6 vs 13.0 us, 512 tokens
// 18.8 vs 13.0 us, 1000 tokens 33 vs 16 us), so larger batches take the three
// launches.
#ifndef MOE_PLAN_SINGLE_MAX_TILES
#define MOE_PLAN_SINGLE_MAX_TILES 4
#endif

// 2048 / THREADS CTAs per SM caps the kernel at 32 registers a thread (a few
// spills at 8 or more keys a lane).  Uncapped, one 1024-thread CTA took the
// whole register file of its SM, so while it ran no dispatch or combine CTA of
// the other buffer set could share that SM; with half the file left free the
// pipelined step is about 2.5 us shorter at 4096 tokens and the plan alone no
// slower.  Smaller CTAs (8 or 16 lanes a token, for small expert counts) take
// a quarter or half of that register file.
template <int EPL, int THREADS, int TT>
__global__ void __launch_bounds__(THREADS, 2048 / THREADS)
route_tile_kernel(const float* __restrict__ logits, int T, int E, int P, int k,
                  const int32_t* __restrict__ rep_off, const int32_t* __restrict__ rep_ids,
                  int32_t* __restrict__ topk_e, float* __restrict__ gates,
                  int32_t* __restrict__ phys, int32_t* __restrict__ tile_hist, int n_tiles,
                  int32_t* __restrict__ local_rank, int32_t* __restrict__ err) {
    extern __shared__ __align__(16) unsigned char smem[];
    grid_dependency_sync();
    allow_dependents();
    MOE_TRACE_SM(tr_route);
    route_tile<EPL, kRouteInRoute, THREADS, TT>(logits, T, E, P, k, rep_off, rep_ids, topk_e, gates, phys,
                                                tile_hist, n_tiles, local_rank, err, smem, blockIdx.x);
}

// One warp: exclusive scan of tile_hist[p, :] in place, counts[p] = column
// total.  Loads bypass L1 (the counts may come from other CTAs of the launch).
constexpr int kScanThreads = 256;
constexpr int kScanBatch = 8;  // chunks of 32 tiles loaded before scanning

__device__ __forceinline__ void scan_column(int32_t* __restrict__ tile_hist, int n_tiles, int p, int lane,
                                            int32_t* __restrict__ counts) {
    int32_t* col = tile_hist + (size_t)p * n_tiles;
    int carry = 0;
    for (int base = 0; base < n_tiles; base += 32 * kScanBatch) {
        int v[kScanBatch];
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u) {
            const int idx = base + u * 32 + lane;
            v[u] = (idx < n_tiles) ? __ldcg(col + idx) : 0;
        }
#pragma unroll
        for (int u = 0; u < kScanBatch; ++u) {
            int incl = v[u];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_up_sync(kFull, incl, off);
                if (lane >= off) incl += o;
            }
            const int idx = base + u * 32 + lane;
            if (idx < n_tiles) col[idx] = carry + incl - v[u];
            carry += __shfl_sync(kFull, incl, 31);
        }
    }
    if (lane == 0) counts[p] = carry;
}

__global__ void __launch_bounds__(kScanThreads)
column_scan_kernel(int32_t* __restrict__ tile_hist, int n_tiles, int P, int32_t* __restrict__ counts) {
    grid_dependency_sync();
    allow_dependents();
    MOE_TRACE_SM(tr_scan);
    MOE_TRACE_MARK(tr_scan, 0);
    const int p = blockIdx.x * (kScanThreads / 32) + (threadIdx.x >> 5);
    if (p < P) scan_column(tile_hist, n_tiles, p, threadIdx.x & 31, counts);
    MOE_TRACE_MARK(tr_scan, 1);
}

// Exclusive scan of counts[0..P) into offs[0..P] in shared memory (whole CTA).
template <int THREADS>
__device__ void block_offsets(const int32_t* __restrict__ counts, int P, int32_t* offs) {
    __shared__ int32_t warp_tot[THREADS / 32];
    const int per = (P + THREADS - 1) / THREADS;
    const int lo = threadIdx.x * per;
    int local = 0;
    for (int i = 0; i < per; ++i)
        if (lo + i < P) local += __ldcg(counts + lo + i);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    // Every warp scans the warp totals with shuffles and takes its base.
    int tot = (lane < THREADS / 32) ? warp_tot[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFull, tot, off);
        if (lane >= off) tot += o;
    }
    const int wbase = __shfl_sync(kFull, tot, warp) - warp_tot[warp];
    int run = wbase + incl - local;
    for (int i = 0; i < per; ++i) {
        if (lo + i < P) {
            offs[lo + i] = run;
            run += __ldcg(counts + lo + i);
        }
    }
    if (threadIdx.x == THREADS - 1) offs[P] = wbase + incl;
    __syncthreads();
}

constexpr int kAssignThreads = 256;

__global__ void __launch_bounds__(kAssignThreads)
assign_kernel(const int32_t* __restrict__ phys, const int32_t* __restrict__ tile_hist, int n_tiles, int tt,
              const int32_t* __restrict__ local_rank, const int32_t* __restrict__ counts, int T, int P,
              int k, int32_t* __restrict__ offsets, int32_t* __restrict__ slot,
              int32_t* __restrict__ src_token, int32_t* __restrict__ src_k, int32_t* __restrict__ err) {
    extern __shared__ int32_t offs[];  // [P+1]
    grid_dependency_sync();
    allow_dependents();
    MOE_TRACE_SM(tr_assign);
    MOE_TRACE_MARK(tr_assign, 0);
    const int n = T * k;
    const int it = blockIdx.x * kAssignThreads + threadIdx.x;
    // Loads that do not depend on the offsets go out before the block scan.
    int p = -1, base = 0, rank = 0;
    if (it < n) {
        p = phys[it];
        rank = local_rank[it];
        if (p >= 0 && p < P) base = tile_hist[(size_t)p * n_tiles + (it / k) / tt];
    }
    block_offsets<kAssignThreads>(counts, P, offs);
    MOE_TRACE_MARK(tr_assign, 1);
    if (blockIdx.x == 0)
        for (int q = threadIdx.x; q <= P; q += kAssignThreads) offsets[q] = offs[q];
    if (it >= n) {
        MOE_TRACE_MARK(tr_assign, 2);
        return;
    }
    const int t = it / k;
    const int j = it - t * k;
    int r = -1;
    if (p >= 0 && p < P) r = offs[p] + base + rank;
    if (r < 0 || r >= n) {
        set_error(err, MOE_DEVERR_SLOT);
        slot[it] = -1;
        return;
    }
    slot[it] = r;
    src_token[r] = t;
    src_k[r] = j;
}

// The single-launch tail, run by one CTA once every tile is routed: column
// scans (one thread per expert; at most MOE_PLAN_SINGLE_MAX_TILES entries
// each), offsets, and the placement of every (t, j) copy.  Counts land in
// shared memory (scanned in place into offsets) and, when they fit
// (col_smem), so do the tile bases.  Data written by other CTAs is read with
// L1-bypassing loads.  The physical expert and in-tile rank of each thread's
// first kTailPrefetch copies are loaded together with the columns, so the
// tail waits for one round trip to L2 instead of two.
constexpr int kTailPrefetch = 2;

__device__ __forceinline__ void place_copy(int it, int p, int rank, int k, int P, int n, int n_tiles,
                                           const int32_t* offs, const int32_t* colpre, int col_smem,
                                           const int32_t* __restrict__ tile_hist, int32_t* __restrict__ slot,
                                           int32_t* __restrict__ src_token, int32_t* __restrict__ src_k,
                                           int32_t* __restrict__ err) {
    const int t = it / k;
    const int j = it - t * k;
    int r = -1;
    if (p >= 0 && p < P) {
        const size_t c = (size_t)p * n_tiles + t / kTileTokens;
        r = offs[p] + (col_smem ? colpre[c] : __ldcg(tile_hist + c)) + rank;
    }
    if (r < 0 || r >= n) {
        set_error(err, MOE_DEVERR_SLOT);
        slot[it] = -1;
        return;
    }
    slot[it] = r;
    src_token[r] = t;
    src_k[r] = j;
}

__device__ void plan_tail(int32_t* __restrict__ tile_hist, int n_tiles, int T, int P, int k,
                          const int32_t* __restrict__ phys, const int32_t* __restrict__ local_rank,
                          int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ slot,
                          int32_t* __restrict__ src_token, int32_t* __restrict__ src_k, int32_t* __restrict__ err,
                          unsigned char* smem, int col_smem) {
    int32_t* offs = reinterpret_cast<int32_t*>(smem);  // [P+1], reuses the route scratch
    int32_t* colpre = offs + (P + 1);                   // [P, n_tiles] when col_smem
    const int n = T * k;
    int pre_p[kTailPrefetch], pre_rank[kTailPrefetch];
#pragma unroll
    for (int u = 0; u < kTailPrefetch; ++u) {
        const int it = threadIdx.x + u * kRouteThreads;
        pre_p[u] = (it < n) ? __ldcg(phys + it) : -1;
        pre_rank[u] = (it < n) ? __ldcg(local_rank + it) : 0;
    }
    // Each thread scans a contiguous chunk of columns and keeps the chunk's
    // total in a register, so the scan of the counts into offsets starts at
    // once (a warp scan, one barrier for the warp totals, one to publish).
    const int per = (P + kRouteThreads - 1) / kRouteThreads;
    const int p_lo = threadIdx.x * per;
    const int p_hi = min(P, p_lo + per);
    int chunk = 0;
    for (int p = p_lo; p < p_hi; ++p) {
        int32_t* col = tile_hist + (size_t)p * n_tiles;
        int32_t* dst = col_smem ? colpre + (size_t)p * n_tiles : col;
        int carry = 0;
        for (int base = 0; base < n_tiles; base += 8) {
            int v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) v[u] = (base + u < n_tiles) ? __ldcg(col + base + u) : 0;
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                if (base + u < n_tiles) dst[base + u] = carry;
                carry += v[u];
            }
        }
        counts[p] = carry;
        offs[p] = carry;
        chunk += carry;
    }
    {
        __shared__ int32_t warp_tot[kRouteThreads / 32];
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        int incl = chunk;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(kFull, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        static_assert(kRouteThreads == 32 * 32, "one warp total per lane");
        int tot = warp_tot[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(kFull, tot, off);
            if (lane >= off) tot += o;
        }
        const int total = __shfl_sync(kFull, tot, 31);
        int run = __shfl_sync(kFull, tot, warp) - warp_tot[warp] + incl - chunk;
        for (int p = p_lo; p < p_hi; ++p) {  // this thread's own entries
            const int v = offs[p];
            offs[p] = run;
            offsets[p] = run;
            run += v;
        }
        if (threadIdx.x == 0) {
            offs[P] = total;
            offsets[P] = total;
        }
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kTailPrefetch; ++u) {
        const int it = threadIdx.x + u * kRouteThreads;
        if (it < n)
            place_copy(it, pre_p[u], pre_rank[u], k, P, n, n_tiles, offs, colpre, col_smem, tile_hist, slot,
                       src_token, src_k, err);
    }
    for (int it = threadIdx.x + kTailPrefetch * kRouteThreads; it < n; it += kRouteThreads)
        place_copy(it, __ldcg(phys + it), __ldcg(local_rank + it), k, P, n, n_tiles, offs, colpre, col_smem,
                   tile_hist, slot, src_token, src_k, err);
}

// Single-launch plan for batches of at most MOE_PLAN_SINGLE_MAX_TILES tiles
// when the cluster plan is not available (trace stages 0-5 as route_tile;
// the last CTA adds 6 scans done, 7 end): every CTA routes its tile; the CTA that finishes last
// (atomic ticket, no waiting) then runs the column scans, the offsets and the
// slot assignment for the whole batch, and resets the ticket for the next
// call.  Each CTA fences its writes before taking its ticket, and the last
// one reads the others' results with L1-bypassing loads.
template <int EPL>
__global__ void __launch_bounds__(kRouteThreads)
plan_single_kernel(const float* __restrict__ logits, int T, int E, int P, int k,
                   const int32_t* __restrict__ rep_off, const int32_t* __restrict__ rep_ids,
                   int32_t* __restrict__ topk_e, float* __restrict__ gates, int32_t* __restrict__ phys,
                   int32_t* __restrict__ tile_hist, int n_tiles, int32_t* __restrict__ local_rank,
                   int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ slot,
                   int32_t* __restrict__ src_token, int32_t* __restrict__ src_k, int32_t* __restrict__ err,
                   int32_t* __restrict__ ticket, int col_smem) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int last;
    grid_dependency_sync();
    allow_dependents();
    MOE_TRACE_SM(tr_single);
    route_tile<EPL, kRouteInSingle, kRouteThreads>(logits, T, E, P, k, rep_off, rep_ids, topk_e, gates, phys,
                                                   tile_hist, n_tiles, local_rank, err, smem, blockIdx.x);
    // The barrier orders every thread's writes before thread 0's fence and
    // ticket (fences are cumulative); in the last CTA, thread 0's second fence
    // and the barrier after it order the other CTAs' results before every
    // thread's reads of them.
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        last = (atomicAdd(ticket, 1) == (int)gridDim.x - 1);
        if (last) __threadfence();
    }
    __syncthreads();
    if (!last) return;

    MOE_TRACE_MARK(tr_single, 6);
    plan_tail(tile_hist, n_tiles, T, P, k, phys, local_rank, counts, offsets, slot, src_token, src_k, err, smem,
              col_smem);
    if (threadIdx.x == 0) *ticket = 0;
    MOE_TRACE_MARK(tr_single, 7);
}

// Batches of at most kClusterTiles tiles (the decode regime), launched as one
// thread-block cluster of one CTA per tile of TT tokens: the smallest of 8,
// 16 and 32 that keeps the cluster within the portable 8 CTAs (8 up to 64
// tokens, 16 up to 128), else 32 (up to 16 CTAs).  A CTA routes one token per
// warp, and 32 warps routing at once on one SM take about twice as long per
// arg-max round as eight, so a small batch is spread over more SMs; larger
// clusters of small tiles plan faster from an idle GPU but wait for SMs when
// another stream's kernels fill the GPU.  Every CTA routes its tile
// (the route_tile body) and keeps its per-expert token masks in shared memory;
// after the cluster barrier each CTA reads every tile's masks over
// distributed shared memory, so it knows, per physical expert, the copies in
// earlier tiles (its tile base) and in all tiles (the counts, scanned into the
// offsets), and places its own tile's copies.  No ticket, no single-CTA tail,
// no global tile counts or ranks.  Trace stages 0-5 as route_tile; 6 cluster
// barrier passed, 7 copies placed.
constexpr int kClusterTiles = 16;        // the largest cluster Blackwell schedules
constexpr int kClusterPortableTiles = 8;  // larger clusters need the non-portable attribute

template <int EPL, int TT>
__global__ void __launch_bounds__(32 * TT)
plan_cluster_kernel(const float* __restrict__ logits, int T, int E, int P, int k,
                    const int32_t* __restrict__ rep_off, const int32_t* __restrict__ rep_ids,
                    int32_t* __restrict__ topk_e, float* __restrict__ gates, int32_t* __restrict__ phys,
                    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ slot,
                    int32_t* __restrict__ src_token, int32_t* __restrict__ src_k, int32_t* __restrict__ err) {
    constexpr int THREADS = 32 * TT;  // one warp per token
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int32_t warp_tot[TT];
    grid_dependency_sync();
    allow_dependents();
    MOE_TRACE_SM(tr_single);
    const int tile = (int)cluster_ctarank();  // the grid is one cluster
    route_tile<EPL, kRouteInCluster, THREADS, TT>(logits, T, E, P, k, rep_off, rep_ids, topk_e, gates, phys,
                                                  nullptr, (int)gridDim.x, nullptr, err, smem, tile);
    // route_tile's shared-memory layout: exp table, sel_v (the selected
    // logits, then the gates), sel_e, sel_p [TT k], masks [P], replica
    // offsets [E+1] and ids [P]; then this kernel's arrays.
    const float2* s_exp = reinterpret_cast<const float2*>(smem);
    float* sel_v = reinterpret_cast<float*>(reinterpret_cast<float2*>(smem) + 2 * dword::kExpTableHalf + 1);
    const float* sel_g = sel_v;
    const int32_t* sel_e = reinterpret_cast<const int32_t*>(sel_g + TT * k);
    const int32_t* sel_p = sel_e + TT * k;
    const uint32_t* mask = reinterpret_cast<const uint32_t*>(sel_p + TT * k);
    int32_t* s_base = const_cast<int32_t*>(reinterpret_cast<const int32_t*>(mask + P)) + (E + 1) + P;  // [P]
    int32_t* offs = s_base + P;                                                                         // [P+1]

    // This CTA's masks are complete.  route_tile left its global stores
    // (top-k ids, gates, physical ids) to the placement loop below, so this
    // arrive's release has only shared memory to publish.
    cluster_arrive();
    // The gates, while the other CTAs arrive: the softmax over each token's
    // selected logits (sel_v, read only by the warp of that token's items),
    // kept in sel_v for the placement loop.
    {
        const float g = tile_gate<kRouteInCluster, TT>(T, k, tile * TT, sel_v, s_exp);
        const int kp = k <= 1 ? 1 : 1 << (32 - __clz(k - 1));
        const int itl = (int)threadIdx.x / kp;
        const int ij = (int)threadIdx.x - itl * kp;
        __syncwarp();  // every lane of the token's segment has read sel_v
        if (itl < TT && ij < k && tile * TT + itl < T) sel_v[itl * k + ij] = g;
    }
    // Every tile's masks are complete and visible in the cluster.
    cluster_wait();
    MOE_TRACE_MARK(tr_single, 6);

    // Per physical expert: copies in earlier tiles and in all tiles.  Each
    // thread takes a contiguous chunk of experts and keeps its chunk's total
    // in a register for the scan into offsets.
    const int n_cta = (int)gridDim.x;
    const int per = (P + THREADS - 1) / THREADS;
    const int p_lo = threadIdx.x * per;
    const int p_hi = min(P, p_lo + per);
    int chunk = 0;
    for (int p = p_lo; p < p_hi; ++p) {
        uint32_t m[kClusterTiles];  // all remote loads in flight before the first use
#pragma unroll
        for (int c = 0; c < kClusterTiles; ++c) m[c] = (c < n_cta) ? ld_cluster_shared_u32(mask + p, (uint32_t)c) : 0u;
        int total = 0, before = 0;
#pragma unroll
        for (int c = 0; c < kClusterTiles; ++c) {
            const int cnt = __popc(m[c]);
            before += (c < tile) ? cnt : 0;
            total += cnt;
        }
        s_base[p] = before;
        offs[p] = total;
        if (tile == 0) counts[p] = total;
        chunk += total;
    }
    // Done reading the other CTAs' masks (their values are consumed above, so
    // the loads have completed; waited for before exit).  Nothing is published.
    cluster_arrive_relaxed();
    MOE_TRACE_MARK(tr_single, 7);

    // Exclusive scan of the totals into offs (warp scan, one barrier for the
    // warp totals, one to publish).
    {
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        int incl = chunk;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(kFull, incl, off);
            if (lane >= off) incl += o;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        int tot = lane < TT ? warp_tot[lane] : 0;  // TT warps, one total each
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int o = __shfl_up_sync(kFull, tot, off);
            if (lane >= off) tot += o;
        }
        const int total = __shfl_sync(kFull, tot, 31);
        int run = __shfl_sync(kFull, tot, warp) - warp_tot[warp] + incl - chunk;
        for (int p = p_lo; p < p_hi; ++p) {  // this thread's own entries
            const int v = offs[p];
            offs[p] = run;
            if (tile == 0) offsets[p] = run;
            run += v;
        }
        if (threadIdx.x == 0) {
            offs[P] = total;
            if (tile == 0) offsets[P] = total;
        }
    }
    __syncthreads();
    MOE_TRACE_MARK(tr_single, 8);

    // Place this tile's copies: slot = offset + tile base + in-tile rank; and
    // store the routing results route_tile kept in shared memory.
    const int n = T * k;
    for (int it = threadIdx.x; it < TT * k; it += THREADS) {
        const int itl = it / k;
        const int j = it - itl * k;
        const int t = tile * TT + itl;
        if (t >= T) continue;
        const int p = sel_p[it];
        const size_t o = (size_t)t * k + j;
        topk_e[o] = sel_e[it];
        gates[o] = sel_g[it];
        phys[o] = p;
        int r = -1;
        if (p >= 0 && p < P) r = offs[p] + s_base[p] + __popc(mask[p] & ((1u << itl) - 1u));
        if (r < 0 || r >= n) {
            set_error(err, MOE_DEVERR_SLOT);
            slot[(size_t)t * k + j] = -1;
            continue;
        }
        slot[(size_t)t * k + j] = r;
        src_token[r] = t;
        src_k[r] = j;
    }
    MOE_TRACE_MARK(tr_single, 9);
    cluster_wait();  // no CTA leaves while another may still read its masks
}


constexpr size_t kTailSmemMax = 96 * 1024;
size_t tail_smem(size_t route_smem, int P, int n_tiles, int* col_smem);


template <typename K>
cudaError_t smem_attr(K kernel, size_t smem) {
    if (smem <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
}

template <int EPL>
cudaError_t launch_single(const float* logits, int T, int E, int P, int k, const int32_t* rep_off,
                          const int32_t* rep_ids, int32_t* topk_e, float* gates, int32_t* phys, int32_t* tile_hist,
                          int32_t* local_rank, int32_t* counts, int32_t* offsets, int32_t* slot,
                          int32_t* src_token, int32_t* src_k, int32_t* err, int32_t* ticket, size_t smem,
                          int n_tiles, int urgent, cudaStream_t s) {
    int col_smem = 0;
    const size_t smem1 = tail_smem(smem, P, n_tiles, &col_smem);
    cudaError_t e;
    if ((e = smem_attr(plan_single_kernel<EPL>, smem1)) != cudaSuccess) return e;
    return launch_pdl_at(urgent, plan_single_kernel<EPL>, dim3(n_tiles), dim3(kRouteThreads), smem1, s, logits, T,
                         E, P, k, rep_off, rep_ids, topk_e, gates, phys, tile_hist, n_tiles, local_rank, counts,
                         offsets, slot, src_token, src_k, err, ticket, col_smem);
}

// Dynamic shared memory of route_tile for tiles of `tt` tokens: exp table,
// sel_v / sel_e / sel_p [tt k], masks [P], replica offsets [E+1] and ids [P].
size_t route_smem(int tt, int E, int P, int k) {
    return (2 * dword::kExpTableHalf + 1) * sizeof(float2) +
           (size_t)tt * k * (sizeof(float) + 2 * sizeof(int32_t)) + (size_t)P * sizeof(uint32_t) +
           (size_t)(E + 1 + P) * sizeof(int32_t);
}

template <int EPL, int TT>
cudaError_t launch_cluster(const float* logits, int T, int E, int P, int k, const int32_t* rep_off,
                           const int32_t* rep_ids, int32_t* topk_e, float* gates, int32_t* phys, int32_t* counts,
                           int32_t* offsets, int32_t* slot, int32_t* src_token, int32_t* src_k, int32_t* err,
                           int urgent, cudaStream_t s) {
    const int n_tiles = (T + TT - 1) / TT;
    const size_t smem1 = route_smem(TT, E, P, k) + (size_t)(2 * P + 1) * sizeof(int32_t);  // + tile bases, offsets
    cudaError_t e;
    if ((e = smem_attr(plan_cluster_kernel<EPL, TT>, smem1)) != cudaSuccess) return e;
    if (n_tiles > kClusterPortableTiles &&
        (e = cudaFuncSetAttribute(plan_cluster_kernel<EPL, TT>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                  1)) != cudaSuccess)
        return e;
    return launch_pdl_cluster(urgent, (unsigned)n_tiles, plan_cluster_kernel<EPL, TT>, dim3(n_tiles),
                              dim3(32 * TT), smem1, s, logits, T, E, P, k, rep_off, rep_ids, topk_e, gates, phys,
                              counts, offsets, slot, src_token, src_k, err);
}

// The cluster plan with tiles of TT tokens for `epl` keys a lane.
template <int TT, typename... A>
cudaError_t launch_cluster_epl(int epl, A... a) {
    if (epl <= 1) return launch_cluster<1, TT>(a...);
    if (epl <= 2) return launch_cluster<2, TT>(a...);
    if (epl <= 4) return launch_cluster<4, TT>(a...);
    if (epl <= 8) return launch_cluster<8, TT>(a...);
    if (epl <= 16) return launch_cluster<16, TT>(a...);
    return launch_cluster<32, TT>(a...);
}

template <int EPL, int THREADS, int TT>
cudaError_t launch_route(const float* logits, int T, int E, int P, int k, const int32_t* rep_off,
                         const int32_t* rep_ids, int32_t* topk_e, float* gates, int32_t* phys, int32_t* tile_hist,
                         int32_t* local_rank, int32_t* err, size_t smem, int n_tiles, int urgent, cudaStream_t s) {
    cudaError_t e;
    if ((e = smem_attr(route_tile_kernel<EPL, THREADS, TT>, smem)) != cudaSuccess) return e;
    return launch_pdl_at(urgent, route_tile_kernel<EPL, THREADS, TT>, dim3(n_tiles), dim3(THREADS), smem, s,
                         logits, T, E, P, k, rep_off, rep_ids, topk_e, gates, phys, tile_hist, n_tiles, local_rank,
                         err);
}

// The route kernel for `epl` keys a lane (a power of two up to 32 / 8) and
// tiles of TT tokens (L = THREADS / TT lanes a token).
template <int THREADS, int TT = kTileTokens, typename... A>
cudaError_t launch_route_epl(int epl, A... a) {
    if (epl <= 1) return launch_route<1, THREADS, TT>(a...);
    if (epl <= 2) return launch_route<2, THREADS, TT>(a...);
    if (epl <= 4) return launch_route<4, THREADS, TT>(a...);
    if constexpr (THREADS / TT == 32) {
        if (epl <= 8) return launch_route<8, THREADS, TT>(a...);
        if (epl <= 16) return launch_route<16, THREADS, TT>(a...);
        return launch_route<32, THREADS, TT>(a...);
    } else {
        return launch_route<8, THREADS, TT>(a...);
    }
}

// Shared memory for the single-launch tail: offsets and, when they fit, the
// tile bases; returns the dynamic smem size and whether bases are in smem.
size_t tail_smem(size_t route_smem, int P, int n_tiles, int* col_smem) {
    const size_t tail = (size_t)(P + 1 + (size_t)P * n_tiles) * sizeof(int32_t);
    *col_smem = tail <= kTailSmemMax ? 1 : 0;
    const size_t need = *col_smem ? tail : (size_t)(P + 1) * sizeof(int32_t);
    return route_smem > need ? route_smem : need;
}

}  // namespace

#ifdef MOE_TRACE
int trace_symbols_plan(int kind, void** stamps, void** sms) {
    cudaError_t e = cudaErrorInvalidValue;
    switch (kind) {
        case kTraceRoute:
            e = cudaGetSymbolAddress(stamps, tr_route_t);
            if (e == cudaSuccess) e = cudaGetSymbolAddress(sms, tr_route_sm);
            break;
        case kTraceColumnScan:
            e = cudaGetSymbolAddress(stamps, tr_scan_t);
            if (e == cudaSuccess) e = cudaGetSymbolAddress(sms, tr_scan_sm);
            break;
        case kTraceAssign:
            e = cudaGetSymbolAddress(stamps, tr_assign_t);
            if (e == cudaSuccess) e = cudaGetSymbolAddress(sms, tr_assign_sm);
            break;
        case kTracePlanSingle:
            e = cudaGetSymbolAddress(stamps, tr_single_t);
            if (e == cudaSuccess) e = cudaGetSymbolAddress(sms, tr_single_sm);
            break;

        default:
            break;
    }
    return e == cudaSuccess ? 0 : -1;
}
#endif

cudaError_t launch_plan(const float* logits, int T, int E, int P, int k, const int32_t* rep_off,
                        const int32_t* rep_ids, int32_t* topk_e, float* gates, int32_t* phys,
                        int32_t* tile_hist, int32_t* local_rank, int32_t* counts, int32_t* offsets,
                        int32_t* slot, int32_t* src_token, int32_t* src_k, int32_t* err, int32_t* ticket,
                        cudaStream_t s, uint64_t* launches) {
    const size_t smem = route_smem(kTileTokens, E, P, k);
    const int n_tiles = (T + kTileTokens - 1) / kTileTokens;
    // The plan is latency-bound and on its stream's critical path; bandwidth-
    // bound kernels of other streams (the other buffer set's dispatch and
    // combine) keep HBM busy meanwhile.  At the most urgent priority the block
    // scheduler places the plan's CTAs ahead of their queued CTAs, so the plan
    // is not stretched by waiting for SM slots.
    const int urgent = most_urgent_priority();
    cudaError_t e;
    if (n_tiles <= kClusterTiles && cluster_launch_supported()) {  // needs no ticket and no scratch
        // The smallest tile that keeps the cluster portable (at most 8 CTAs);
        // 32-token tiles beyond that, in up to kClusterTiles CTAs.
        const int epl = (E + 31) / 32;
        if (T <= 8 * kClusterPortableTiles)
            e = launch_cluster_epl<8>(epl, logits, T, E, P, k, rep_off, rep_ids, topk_e, gates, phys, counts,
                                      offsets, slot, src_token, src_k, err, urgent, s);
        else if (T <= 16 * kClusterPortableTiles)
            e = launch_cluster_epl<16>(epl, logits, T, E, P, k, rep_off, rep_ids, topk_e, gates, phys, counts,
                                       offsets, slot, src_token, src_k, err, urgent, s);
        else
            e = launch_cluster_epl<32>(epl, logits, T, E, P, k, rep_off, rep_ids, topk_e, gates, phys, counts,
                                       offsets, slot, src_token, src_k, err, urgent, s);
        if (e == cudaSuccess) {
            *launches += 1;
            return e;
        }
        // A cluster this size that cannot be placed is a launch-time error
        // (nothing was enqueued and the context stays usable): clear it and
        // use the ticket kernel (up to MOE_PLAN_SINGLE_MAX_TILES tiles) or
        // the three launches instead.
        (void)cudaGetLastError();
    }
    if (ticket != nullptr && n_tiles <= MOE_PLAN_SINGLE_MAX_TILES) {
        const int epl = (E + 31) / 32;
#define MOE_SINGLE_CASE(N)                                                                                      \
    e = launch_single<N>(logits, T, E, P, k, rep_off, rep_ids, topk_e, gates, phys, tile_hist, local_rank, counts, \
                         offsets, slot, src_token, src_k, err, ticket, smem, n_tiles, urgent, s)
        if (epl <= 1) MOE_SINGLE_CASE(1);
        else if (epl <= 2) MOE_SINGLE_CASE(2);
        else if (epl <= 4) MOE_SINGLE_CASE(4);
        else if (epl <= 8) MOE_SINGLE_CASE(8);
        else if (epl <= 16) MOE_SINGLE_CASE(16);
        else MOE_SINGLE_CASE(32);
#undef MOE_SINGLE_CASE
        if (e == cudaSuccess) *launches += 1;
        return e;
    }

    // Three launches.  Lanes per token: route_lanes; tokens per tile:
    // route_tile_tokens (16 for mid-size batches of whole-warp tokens).  The
    // tile-count scratch has route_tiles(T) columns.
    const int L = route_lanes(E, k);
    const int tt = route_tile_tokens(T, E, k);
    const int tiles = (T + tt - 1) / tt;
    const size_t rsmem = route_smem(tt, E, P, k);
    const int epl = (E + L - 1) / L;
    if (L == 8)
        e = launch_route_epl<256>(epl, logits, T, E, P, k, rep_off, rep_ids, topk_e, gates, phys, tile_hist,
                                  local_rank, err, rsmem, tiles, urgent, s);
    else if (L == 16)
        e = launch_route_epl<512>(epl, logits, T, E, P, k, rep_off, rep_ids, topk_e, gates, phys, tile_hist,
                                  local_rank, err, rsmem, tiles, urgent, s);
    else if (tt == kMidTileTokens)
        e = launch_route_epl<32 * kMidTileTokens, kMidTileTokens>(epl, logits, T, E, P, k, rep_off, rep_ids,
                                                                   topk_e, gates, phys, tile_hist, local_rank, err,
                                                                   rsmem, tiles, urgent, s);
    else
        e = launch_route_epl<kRouteThreads>(epl, logits, T, E, P, k, rep_off, rep_ids, topk_e, gates, phys,
                                            tile_hist, local_rank, err, rsmem, tiles, urgent, s);
    if (e != cudaSuccess) return e;
    *launches += 1;

    e = launch_pdl_at(urgent, column_scan_kernel, dim3((P + 7) / 8), dim3(kScanThreads), 0, s, tile_hist, tiles,
                      P, counts);
    if (e != cudaSuccess) return e;
    *launches += 1;

    const int n = T * k;
    e = launch_pdl_at(urgent, assign_kernel, dim3((n + kAssignThreads - 1) / kAssignThreads),
                      dim3(kAssignThreads), (P + 1) * sizeof(int32_t), s, phys, (const int32_t*)tile_hist, tiles, tt,
                      (const int32_t*)local_rank, (const int32_t*)counts, T, P, k, offsets, slot, src_token,
                      src_k, err);
    if (e != cudaSuccess) return e;
    *launches += 1;
    return cudaSuccess;
}

}  // namespace moe
