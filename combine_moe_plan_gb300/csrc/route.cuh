// route.cuh -- routing of one 32-token tile: the body every plan kernel
// runs per CTA (top-k by segment arg-max, gates from float pairs, replica
// pick, per-expert token masks, tile counts and in-tile ranks), with its key
// mapping and lane helpers.  Included once, by plan.cu, after the trace
// buffers tr_route and tr_single are defined.
#pragma once

#include <climits>
#include <cstdint>

#include "dword.cuh"
#include "moe_internal.h"
#include "ptx.cuh"
#include "trace.cuh"

namespace moe {
namespace {

// The two largest keys of a lane that are not yet taken (bit r of `taken`
// marks slot r) and their slots (lower slot first among equal keys); k2 = 0
// if the lane has fewer than two such keys above 0.
template <int N>
__device__ __forceinline__ void lane_top2(const uint32_t (&key)[N], uint32_t taken, uint32_t& k1, int& r1,
                                          uint32_t& k2, int& r2) {
    k1 = 0u;
    r1 = 0;
    k2 = 0u;
    r2 = 0;
#pragma unroll
    for (int r = 0; r < N; ++r) {
        const uint32_t v = ((taken >> r) & 1u) ? 0u : key[r];
        if (v > k1) {
            k2 = k1;
            r2 = r1;
            k1 = v;
            r1 = r;
        } else if (v > k2) {
            k2 = v;
            r2 = r;
        }
    }
}

// Which kernel a route_tile call belongs to (its trace slice; the cluster
// plan keeps tile counts and ranks in shared memory instead of writing them).
constexpr int kRouteInRoute = 0, kRouteInSingle = 1, kRouteInCluster = 2;

#ifdef MOE_TRACE
// Stage stamps of route_tile go to the slice of the kernel that called it.
template <int WHERE>
__device__ __forceinline__ TraceSlice route_slice() {
    return WHERE == kRouteInRoute ? tr_route_t : tr_single_t;
}
#define ROUTE_MARK(stage) trace_mark(route_slice<WHERE>(), (stage))
#else
#define ROUTE_MARK(stage) ((void)0)
#endif

constexpr int kRouteThreads = 32 * kTileTokens;  // one warp per token of the tile


// Monotone map of finite floats onto uint32 (a < b  <=>  key(a) < key(b));
// -0 is folded onto +0 first, so equal values give equal keys.  Every finite
// value maps above 0.
__device__ __forceinline__ uint32_t order_key(float f) {
    uint32_t b = __float_as_uint(f);
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Inverse of order_key (a -0 logit comes back as +0).
__device__ __forceinline__ float key_value(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// The gate of this thread's item (token itl = threadIdx.x / kp of the tile,
// j = threadIdx.x mod kp; 0 for a thread without an item), from the tile's
// selected logits sel_v [TT k] and the exp table in shared memory.
// Warp-collective in the first TT kp threads (whole warps).
template <int WHERE, int TT>
__device__ __forceinline__ float tile_gate(int T, int k, int t0, const float* sel_v, const float2* s_exp) {
    // ---- gates: g_j = exp(l_j - l_0) / sum_i exp(l_i - l_0), rounded once
    // to fp32.  Each token's k items sit in one segment of kp lanes (kp the
    // power of two >= k, so a segment never straddles a warp).  Each lane
    // forms d = l_j - l_0 exactly as a pair of floats and e_j = exp(d) as a
    // pair; a butterfly over the segment sums the pairs (every lane ends with
    // the same s: the pair sum is commutative); each lane divides e_j by s and
    // keeps the high float if Ziv's test shows it is the correctly rounded
    // quotient.  A token with an item the pairs cannot decide, or with
    // l_j - l_0 < -64, is redone in fp64 as e_j = exp(d) with e_0 = 1,
    // s = sum over j ascending and g_j = (float)(e_j / s). ----
    const int kp = k <= 1 ? 1 : 1 << (32 - __clz(k - 1));  // TT kp <= the CTA's threads
    const int itl = (int)threadIdx.x / kp;  // token within the tile (>= TT: no item)
    const int ij = (int)threadIdx.x - itl * kp;
    const int it = itl * k + ij;
    const bool item_ok = itl < TT && ij < k && t0 + itl < T;
    float g = 0.0f;
    bool slow = false;
    // Only the first TT kp threads hold items; warps past them skip the stage.
    // The test is per warp (TT kp may be below 32), so a warp that enters
    // enters whole and its full-mask shuffles see every lane.
    const bool gate_warp = ((int)threadIdx.x & ~31) < TT * kp;
    if (gate_warp) {
        dword::dw e = {0.0f, 0.0f};
        if (item_ok) {
            const dword::dw d = dword::two_sum(sel_v[it], -sel_v[itl * k]);
            if (d.h == 0.0f)
                e = {1.0f, 0.0f};  // j == 0, or a tie with the top logit
            else if (d.h >= -64.0f)
                e = dword::exp_dw(d.h, d.l, s_exp);
            else
                slow = true;  // far below the top logit (or not finite)
        }
        dword::dw s = e;
        for (int off = 1; off < kp; off <<= 1) {
            const dword::dw o = {__shfl_xor_sync(kFull, s.h, off), __shfl_xor_sync(kFull, s.l, off)};
            s = dword::dw_add(s, o);
        }
        if (item_ok && !slow) {
            const dword::dw q = dword::dw_div(e, s);
            g = q.h;
            slow = !dword::rounds_safely(q);
        }
    }
    ROUTE_MARK(2);
    const unsigned slow_lanes = gate_warp ? __ballot_sync(kFull, slow) : 0u;
    if (slow_lanes != 0u) {  // warp-uniform; rare
        const int seg = (int)(threadIdx.x & 31) & ~(kp - 1);
        const unsigned seg_bits = (kp == 32 ? 0xffffffffu : ((1u << kp) - 1u)) << seg;
        const bool redo = (slow_lanes & seg_bits) != 0u && item_ok;
        double e64 = 0.0;
        if (redo) e64 = (ij == 0) ? 1.0 : exp((double)sel_v[it] - (double)sel_v[itl * k]);
        double s64 = 0.0;
        for (int jj = 0; jj < k; ++jj) s64 += __shfl_sync(kFull, e64, seg + jj);
        if (redo) g = (float)(e64 / s64);
    }
    ROUTE_MARK(3);
    return g;
}

// Route one tile of TT tokens (the body every plan kernel runs per CTA) with
// a CTA of THREADS = TT L threads: each token's top-k runs on a segment of L
// lanes (L = 32: a whole warp; 16 or 8 when the experts fit in at most 8 keys
// a lane, so that small expert counts do not occupy a whole warp per token).
// Tiles are 32 tokens (one mask word) except in the cluster plan, which
// spreads a small batch over more SMs with tiles of 8 or 16 tokens.
// Trace stages: 0 start, 1 top-k done, 2 gates from pairs done, 3 fp64
// fallback done, 4 replicas and masks done, 5 tile counts and ranks written.
template <int EPL, int WHERE, int THREADS, int TT = kTileTokens>  // EPL = logits per lane = ceil(E / L)
__device__ __forceinline__ void route_tile(const float* __restrict__ logits, int T, int E, int P, int k,
                                           const int32_t* __restrict__ rep_off,
                                           const int32_t* __restrict__ rep_ids, int32_t* __restrict__ topk_e,
                                           float* __restrict__ gates, int32_t* __restrict__ phys,
                                           int32_t* __restrict__ tile_hist, int n_tiles,
                                           int32_t* __restrict__ local_rank, int32_t* __restrict__ err,
                                           unsigned char* smem, int tile) {
    constexpr int L = THREADS / TT;  // lanes per token
    static_assert(L == 8 || L == 16 || L == 32, "8, 16 or 32 lanes per token");
    static_assert(TT == 8 || TT == 16 || TT == 32, "8, 16 or 32 tokens per tile (bits of a mask word)");
    float2* s_exp = reinterpret_cast<float2*>(smem);                             // exp(m / 512) table
    float* sel_v = reinterpret_cast<float*>(s_exp + 2 * dword::kExpTableHalf + 1);  // [TT*k]
    int32_t* sel_e = reinterpret_cast<int32_t*>(sel_v + TT * k);  // [TT*k]
    int32_t* sel_p = sel_e + TT * k;                               // [TT*k]
    uint32_t* mask = reinterpret_cast<uint32_t*>(sel_p + TT * k);  // [P]
    int32_t* s_off = reinterpret_cast<int32_t*>(mask + P);                 // [E+1] replica CSR
    int32_t* s_ids = s_off + (E + 1);                                       // [P]

    ROUTE_MARK(0);
    // The exp table and the replica map go to shared memory by asynchronous
    // copies (no registers held, no wait) while the logits are loaded; they
    // are waited for before the barrier that ends the top-k.
    for (int i = threadIdx.x; i <= 2 * dword::kExpTableHalf; i += THREADS)
        cp_async8(s_exp + i, dword::kExpTable + i);
    if (rep_off != nullptr) {
        for (int i = threadIdx.x; i <= E; i += THREADS) cp_async4(s_off + i, rep_off + i);
        for (int i = threadIdx.x; i < P; i += THREADS) cp_async4(s_ids + i, rep_ids + i);
    }
    const int tl = threadIdx.x / L;  // this segment's token within the tile
    const int sl = threadIdx.x % L;  // lane within the segment
    const int t0 = tile * TT;
    const int t = t0 + tl;

    // ---- top-k of token t: k rounds of segment arg-max, ties -> lower id ----
    // Logits become order-preserving unsigned keys (-0 folded onto +0 so that
    // equal floats give equal keys); lane s of the segment holds experts
    // s, s + L, s + 2L, ...  Each lane caches its two largest keys; a round
    // is one max-reduction of the lanes' first keys over the segment and one
    // min-reduction of the expert id among the lanes holding the maximum,
    // after which the winning lane marks the slot taken and promotes its
    // second key (rescanning only when it has none left).  Key 0 sits below
    // every finite logit and marks padding.  Lane j keeps the j-th winner and
    // its key, whose inverse is the selected logit.  Every lane runs the
    // rounds (a token past T has only padding keys and writes nothing), so
    // the segment butterflies below always see a converged warp.
    {
        const bool tok_ok = t < T;
        const float* row = logits + (size_t)(tok_ok ? t : t0) * E;
        uint32_t key[EPL];
#pragma unroll
        for (int r = 0; r < EPL; ++r) {
            const int e = r * L + sl;
            key[r] = (tok_ok && e < E) ? order_key(__ldg(row + e)) : 0u;
        }
        uint32_t taken = 0u, k1, k2;
        int r1, r2;
        lane_top2(key, taken, k1, r1, k2, r2);
        uint32_t cand = (uint32_t)(r1 * L + sl);
        int my_e = 0;
        uint32_t my_key = 0u;
        for (int j = 0; j < k; ++j) {
            uint32_t m;
            int win;
            if (L == 32) {  // whole warp: redux.sync (26 cycles on GB300)
                m = __reduce_max_sync(kFull, k1);
                win = (int)__reduce_min_sync(kFull, (k1 == m) ? cand : (uint32_t)INT_MAX);
            } else {
                // A segment-masked redux.sync takes about 170 cycles here, so
                // the segment reduces (key, ~id) packed in 64 bits with one
                // xor butterfly: the largest key, then the smallest id.
                uint64_t kv = ((uint64_t)k1 << 32) | (uint64_t)(0xffffffffu - cand);
#pragma unroll
                for (int off = L / 2; off > 0; off >>= 1) {
                    const uint64_t o = __shfl_xor_sync(kFull, kv, off);
                    kv = o > kv ? o : kv;
                }
                m = (uint32_t)(kv >> 32);
                win = (int)(0xffffffffu - (uint32_t)kv);
            }
            if (win >= E) win = 0;  // only reachable with NaN logits (outside the domain)
            if (sl == (win & (L - 1))) {
                taken |= 1u << r1;
                if (k2 != 0u) {
                    k1 = k2;
                    r1 = r2;
                    k2 = 0u;
                } else {
                    lane_top2(key, taken, k1, r1, k2, r2);
                }
                cand = (uint32_t)(r1 * L + sl);
            }
            if (sl == j) {
                my_e = win;
                my_key = m;
            }
        }
        if (tok_ok && sl < k) {
            sel_v[tl * k + sl] = key_value(my_key);
            sel_e[tl * k + sl] = my_e;
        }
    }
    for (int p = threadIdx.x; p < P; p += THREADS) mask[p] = 0u;
    cp_async_wait_all();
    __syncthreads();
    ROUTE_MARK(1);

    const int kp = k <= 1 ? 1 : 1 << (32 - __clz(k - 1));  // TT kp <= THREADS (host's choice of L)
    const int itl = (int)threadIdx.x / kp;  // token within the tile (>= 32: no item)
    const int ij = (int)threadIdx.x - itl * kp;
    const int it = itl * k + ij;
    const bool item_ok = itl < TT && ij < k && t0 + itl < T;
    // The cluster plan computes the gates after its cluster barrier's arrive
    // (tile_gate there), where they hide behind the wait for the other CTAs.
    float g = 0.0f;
    if (WHERE != kRouteInCluster) g = tile_gate<WHERE, TT>(T, k, t0, sel_v, s_exp);
    if (item_ok) {
        const int tt = t0 + itl;
        const int e = sel_e[it];
        int p = e;
        if (rep_off != nullptr) {
            const int lo = s_off[e];
            const int n = s_off[e + 1] - lo;
            if (n < 1 || lo < 0 || lo + n > P) {
                p = -1;
            } else {
                p = s_ids[lo + tt % n];
                if (p < 0 || p >= P) p = -1;
            }
            if (p < 0) set_error(err, MOE_DEVERR_REPLICA);
        }
        if (WHERE != kRouteInCluster) {  // the cluster plan stores these after its barrier
            const size_t o = (size_t)tt * k + ij;
            topk_e[o] = e;
            gates[o] = g;
            phys[o] = p;
        }
        sel_p[it] = p;
        if (p >= 0) {
            const uint32_t bit = 1u << itl;
            const uint32_t old = atomicOr(&mask[p], bit);
            if (old & bit) set_error(err, MOE_DEVERR_DUPLICATE);
        }
    }
    __syncthreads();
    ROUTE_MARK(4);

    // ---- tile histogram (expert-major) and in-tile ranks ----
    if (WHERE != kRouteInCluster) {
        for (int p = threadIdx.x; p < P; p += THREADS)
            tile_hist[(size_t)p * n_tiles + tile] = __popc(mask[p]);
        if (item_ok) {
            const int p = sel_p[it];
            local_rank[(size_t)(t0 + itl) * k + ij] = (p >= 0) ? __popc(mask[p] & ((1u << itl) - 1u)) : 0;
        }
    }
    ROUTE_MARK(5);
}

}  // namespace
}  // namespace moe
