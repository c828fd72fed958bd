// ep.cu -- the expert-parallel split of the pool over R ranks: ownership,
// receive layout, the transfer schedule (host), and the pull exchange
// (device).
//
// StrataCL analysis, section 3.5 (Workload-balanced NPU-core Partitioning):
// token placement -> expert-window aggregation -> peer-window partition; each
// peer's payload cut into transfer units of at most S_t rows, unit cost
// alpha_t + bytes / beta_t per tier, min-makespan under a per-peer fan-out cap
// per stripe, solved by an LPT-style list scheduler that outputs a task list
// per core.  Section 3.4 (Full-mesh): a collective is a set of remote-slice
// tuples <peer, src, dst, bytes>; data-movement collectives pull -- each rank
// reads remote slices into its own buffer, no producer-consumer handshake.
//
// GPU mapping of the pull: one CTA per (core, puller); a core walks its unit
// list in order, and every thread of the CTA streams its share of each
// unit's contiguous byte range with 16-byte loads (four in flight per thread)
// and 16-byte stores.  A unit is one contiguous run of rows in both buffers
// (a piece of one peer's window of one expert), so a plane of a unit is a
// plain memcpy; the schedule decides which core moves what, in which order.
#include <unistd.h>

#include <algorithm>
#include <atomic>
#include <condition_variable>
#include <cstring>
#include <functional>
#include <mutex>
#include <thread>
#include <vector>

#include "moe_ep.h"
#include "moe_internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace moe {
namespace {

// First expert of rank d: the smallest p with floor(p * R / P) >= d, i.e.
// ceil(d * P / R).
inline int32_t rank_first_expert(int32_t d, int32_t R, int32_t P) {
    return (int32_t)(((int64_t)d * P + R - 1) / R);
}

inline int32_t expert_owner(int32_t p, int32_t R, int32_t P) { return (int32_t)(((int64_t)p * R) / P); }

int check_group(int32_t R, int32_t P) {
    if (R < 1 || R > MOE_EP_MAX_RANKS || P < 1 || P > 4096) return MOE_ERR_SIZE;
    return MOE_OK;
}

int check_desc(const moe_ep_desc* d) {
    if (d == nullptr) return MOE_ERR_NULL;
    int rc = check_group(d->R, d->P);
    if (rc != MOE_OK) return rc;
    if (d->cores < 1 || d->cores > 4096) return MOE_ERR_SIZE;
    for (int t = 0; t < 2; ++t)
        if (d->fanout_cap[t] < 1 || d->unit_rows[t] < 1 || d->unit_rows[t] > (1 << 20) || d->alpha_ns[t] < 0 ||
            d->alpha_ns[t] > ((int64_t)1 << 40) || d->beta_gbs[t] < 1)
            return MOE_ERR_SIZE;
    return MOE_OK;
}

// ---------------------------------------------------------------- pull ----

constexpr int kPullThreads = 512;
constexpr int kPullUnroll = 4;  // 16-byte loads in flight per thread

struct PullPlanes {
    const char* src[2][MOE_EP_MAX_RANKS];
    char* dst[2][MOE_EP_MAX_RANKS];
    int64_t src_rows[2][MOE_EP_MAX_RANKS];
    int64_t dst_rows[2][MOE_EP_MAX_RANKS];
    int64_t row_bytes[2];
    int32_t n_planes;
};

// Copy n16 16-byte words from src to dst with the whole CTA.
__device__ __forceinline__ void cta_copy16(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n16) {
    constexpr int64_t kStep = (int64_t)kPullThreads * kPullUnroll;
    int64_t j = threadIdx.x;
    for (; j + (kPullUnroll - 1) * kPullThreads < n16; j += kStep) {
        uint4 v[kPullUnroll];
#pragma unroll
        for (int u = 0; u < kPullUnroll; ++u) v[u] = ld_stream16(src + j + u * kPullThreads);
#pragma unroll
        for (int u = 0; u < kPullUnroll; ++u) st16(dst + j + u * kPullThreads, v[u]);
    }
    for (; j < n16; j += kPullThreads) st16(dst + j, ld_stream16(src + j));
}

__global__ void __launch_bounds__(kPullThreads)
ep_pull_kernel(const moe_ep_unit* __restrict__ units, const int32_t* __restrict__ core_off, int32_t n_units,
               int32_t R, int32_t C, int32_t first_puller, const PullPlanes pl, int32_t* __restrict__ err) {
    grid_dependency_sync();
    allow_dependents();
    const int c = blockIdx.x;
    const int i = blockIdx.y;
    const int r = first_puller + i;
    const int32_t* co = core_off + (size_t)i * (C + 1);
    const int32_t b = co[c], e = co[c + 1];
    if (b < 0 || e > n_units || b > e) {
        if (threadIdx.x == 0) set_error(err, MOE_DEVERR_UNIT);
        return;
    }
    for (int32_t k = b; k < e; ++k) {
        const moe_ep_unit u = units[k];
        bool ok = u.peer >= 0 && u.peer < R && u.rows >= 0 && u.src_row >= 0 && u.dst_row >= 0;
        for (int p = 0; p < pl.n_planes && ok; ++p)
            ok = (int64_t)u.src_row + u.rows <= pl.src_rows[p][u.peer] &&
                 (int64_t)u.dst_row + u.rows <= pl.dst_rows[p][r] &&
                 (u.rows == 0 || (pl.src[p][u.peer] != nullptr && pl.dst[p][r] != nullptr));
        if (!ok) {  // uniform over the CTA: every thread read the same unit
            if (threadIdx.x == 0) set_error(err, MOE_DEVERR_UNIT);
            continue;
        }
        for (int p = 0; p < pl.n_planes; ++p) {
            const int64_t rb = pl.row_bytes[p];
            cta_copy16(reinterpret_cast<const uint4*>(pl.src[p][u.peer] + (int64_t)u.src_row * rb),
                       reinterpret_cast<uint4*>(pl.dst[p][r] + (int64_t)u.dst_row * rb), (int64_t)u.rows * rb / 16);
        }
    }
}

// ------------------------------------------------------------ workers ----

// A few host threads kept for the scheduler's group calls, so that a call
// does not pay for creating threads.  Created on first use and kept until the
// process exits (detached: nothing is joined at exit).  One group call uses
// them at a time; a call that finds them busy, or a process forked after they
// were created (the child has none of them), runs its tasks on its own thread.
class Workers {
  public:
    static Workers& get() {
        static Workers* w = new Workers();  // never destroyed
        return *w;
    }

    // task(i) for every i in [0, n), on the workers and the calling thread;
    // returns once all have finished.  task must not throw.
    void run(int n, const std::function<void(int)>& task) {
        std::unique_lock<std::mutex> busy(run_mu_, std::try_to_lock);
        if (!busy.owns_lock() || getpid() != owner_pid_ || threads_ == 0) {
            for (int i = 0; i < n; ++i) task(i);
            return;
        }
        {
            std::lock_guard<std::mutex> lock(mu_);
            task_ = &task;
            n_ = n;
            next_ = 0;
            running_ = threads_;
            ++generation_;
        }
        cv_work_.notify_all();
        drain();
        std::unique_lock<std::mutex> lock(mu_);
        cv_done_.wait(lock, [&] { return running_ == 0; });
        task_ = nullptr;
    }

  private:
    Workers() : owner_pid_(getpid()) {
        const unsigned hw = std::thread::hardware_concurrency();
        const int want = (int)std::min<unsigned>(hw > 1 ? hw - 1 : 0, 15);
        for (int i = 0; i < want; ++i) {
            try {
                std::thread(&Workers::loop, this).detach();
                ++threads_;
            } catch (...) {
                break;  // fewer workers; the caller takes the rest
            }
        }
    }

    void drain() {
        for (int i = next_++; i < n_; i = next_++) (*task_)(i);
    }

    void loop() {
        uint64_t seen = 0;
        for (;;) {
            {
                std::unique_lock<std::mutex> lock(mu_);
                cv_work_.wait(lock, [&] { return generation_ != seen; });
                seen = generation_;
            }
            drain();
            std::lock_guard<std::mutex> lock(mu_);
            if (--running_ == 0) cv_done_.notify_all();
        }
    }

    std::mutex run_mu_, mu_;
    std::condition_variable cv_work_, cv_done_;
    const std::function<void(int)>* task_ = nullptr;
    int n_ = 0;
    std::atomic<int> next_{0};
    int running_ = 0;
    uint64_t generation_ = 0;
    int threads_ = 0;
    const pid_t owner_pid_;
};

// ------------------------------------------------------------ schedule ----

// Window starts of every rank from the counts.  pool[s * (P + 1) + p]: expert
// p's first row in rank s's pool (the plan's exclusive scan); recv[s * P + p]:
// s's first row of expert p in its owner's receive buffer.
struct Windows {
    int32_t R = 0, P = 0;
    std::vector<int64_t> pool, recv;

    int build(int32_t R_, int32_t P_, const int32_t* counts) {
        R = R_;
        P = P_;
        pool.assign((size_t)R * (P + 1), 0);
        recv.assign((size_t)R * P, 0);
        for (int32_t s = 0; s < R; ++s) {
            int64_t acc = 0;
            for (int32_t p = 0; p < P; ++p) {
                pool[(size_t)s * (P + 1) + p] = acc;
                acc += counts[(size_t)s * P + p];
            }
            pool[(size_t)s * (P + 1) + P] = acc;
            if (acc > INT32_MAX) return MOE_ERR_SIZE;
        }
        for (int32_t d = 0; d < R; ++d) {
            int64_t row = 0;
            for (int32_t p = rank_first_expert(d, R, P); p < rank_first_expert(d + 1, R, P); ++p)
                for (int32_t s = 0; s < R; ++s) {
                    recv[(size_t)s * P + p] = row;
                    row += counts[(size_t)s * P + p];
                }
            if (row > INT32_MAX) return MOE_ERR_SIZE;
        }
        return MOE_OK;
    }
};

struct Schedule {
    std::vector<moe_ep_unit> units;  // grouped by core, each core's list in assignment order
    std::vector<int32_t> core_off;   // [C + 1]
    int64_t makespan = 0;
};

int check_schedule_args(const moe_ep_desc* desc, int32_t direction, const int32_t* counts, int64_t row_bytes,
                        int32_t max_units) {
    int rc = check_desc(desc);
    if (rc != MOE_OK) return rc;
    if ((direction != 0 && direction != 1) || row_bytes < 1 || row_bytes > ((int64_t)1 << 24) || max_units < 0)
        return MOE_ERR_SIZE;
    for (size_t i = 0; i < (size_t)desc->R * desc->P; ++i)
        if (counts[i] < 0) return MOE_ERR_SIZE;
    return MOE_OK;
}

// The schedule of one puller: units in ascending destination row with their
// costs (ps), longest first (equal costs in that order), each to the
// least-loaded eligible core (equal loads: the lower core) under the fan-out
// cap.
void schedule_one(const moe_ep_desc& desc, const Windows& w, const int32_t* counts, int32_t direction,
                  int32_t puller, int64_t row_bytes, Schedule* out) {
    const int32_t R = desc.R, P = desc.P, C = desc.cores;
    auto cost_of = [&](int t, int64_t rows) {
        return desc.alpha_ns[t] * 1000 + rows * row_bytes * 1000 / desc.beta_gbs[t];
    };
    const int64_t full_cost[2] = {cost_of(0, desc.unit_rows[0]), cost_of(1, desc.unit_rows[1])};

    // 1. units in ascending destination row.  A full unit (S_t rows) of tier t
    // costs full_cost[t], so the full units of a tier are already in order
    // among themselves; only the shorter last pieces of windows need sorting.
    std::vector<moe_ep_unit> u;
    std::vector<int32_t> full[2];
    struct Key {
        int64_t cost;
        int32_t idx;
    };
    std::vector<Key> tails;
    auto cut = [&](int32_t peer, int64_t src0, int64_t dst0, int64_t n) {
        const int t = peer == puller ? 0 : 1;
        const int64_t S = desc.unit_rows[t];
        for (int64_t at = 0; at < n; at += S) {
            const int64_t rows = std::min(S, n - at);
            const int32_t idx = (int32_t)u.size();
            u.push_back(moe_ep_unit{peer, (int32_t)(src0 + at), (int32_t)(dst0 + at), (int32_t)rows});
            if (rows == S)
                full[t].push_back(idx);
            else
                tails.push_back(Key{cost_of(t, rows), idx});
        }
    };
    if (direction == 0) {
        for (int32_t p = rank_first_expert(puller, R, P); p < rank_first_expert(puller + 1, R, P); ++p)
            for (int32_t s = 0; s < R; ++s)
                cut(s, w.pool[(size_t)s * (P + 1) + p], w.recv[(size_t)s * P + p], counts[(size_t)s * P + p]);
    } else {
        for (int32_t p = 0; p < P; ++p)
            cut(expert_owner(p, R, P), w.recv[(size_t)puller * P + p], w.pool[(size_t)puller * (P + 1) + p],
                counts[(size_t)puller * P + p]);
    }
    const int32_t nu = (int32_t)u.size();

    // 2. longest first, equal costs in enumeration order: merge the two runs
    // of full units with the sorted tails.
    auto later = [](const Key& a, const Key& b) { return a.cost != b.cost ? a.cost < b.cost : a.idx > b.idx; };
    std::sort(tails.begin(), tails.end(), [&](const Key& a, const Key& b) { return later(b, a); });
    std::vector<Key> order;
    order.reserve(nu);
    {
        size_t i0 = 0, i1 = 0, it = 0;
        while (order.size() < (size_t)nu) {
            Key best{-1, -1};
            int from = -1;
            if (i0 < full[0].size()) best = Key{full_cost[0], full[0][i0]}, from = 0;
            if (i1 < full[1].size()) {
                const Key c{full_cost[1], full[1][i1]};
                if (from < 0 || later(best, c)) best = c, from = 1;
            }
            if (it < tails.size() && (from < 0 || later(best, tails[it]))) best = tails[it], from = 2;
            order.push_back(best);
            if (from == 0) ++i0;
            else if (from == 1) ++i1;
            else ++it;
        }
    }

    // 3. list scheduling under the fan-out cap.  Cores sit in a min-heap of
    // (load, core) packed into one 128-bit key; a unit takes the first
    // eligible core popped, i.e. the least-loaded eligible core with ties to
    // the lower core.  A core with the longest list is always eligible (its
    // next stripe is still empty), so the search ends.
    using Slot = unsigned __int128;
    auto slot_of = [](int64_t load, int32_t c) { return ((Slot)(uint64_t)load << 32) | (uint32_t)c; };
    std::vector<int32_t> len(C, 0), core_of(nu), pos(nu);
    std::vector<int64_t> load(C, 0);
    std::vector<int32_t> stripe;  // stripe[i * R + q]: cores whose i-th unit is from peer q
    std::vector<Slot> heap(C), held;
    for (int32_t c = 0; c < C; ++c) heap[c] = slot_of(0, c);  // already a heap: ascending
    const std::greater<Slot> above;
    for (int32_t k = 0; k < nu; ++k) {
        const int32_t i = order[k].idx;
        const int32_t q = u[i].peer;
        const int32_t cap = desc.fanout_cap[q == puller ? 0 : 1];
        held.clear();
        int32_t best = -1;
        while (best < 0) {
            std::pop_heap(heap.begin(), heap.end(), above);
            const Slot top = heap.back();
            heap.pop_back();
            const int32_t c = (int32_t)(uint32_t)top;
            const size_t at = (size_t)len[c] * R + q;
            if (at >= stripe.size() || stripe[at] < cap)
                best = c;
            else
                held.push_back(top);
        }
        const size_t at = (size_t)len[best] * R + q;
        if (at >= stripe.size()) stripe.resize(((size_t)len[best] + 1) * R * 2, 0);
        stripe[at] += 1;
        core_of[i] = best;
        pos[i] = len[best];
        len[best] += 1;
        load[best] += order[k].cost;
        held.push_back(slot_of(load[best], best));
        for (const Slot& h : held) {
            heap.push_back(h);
            std::push_heap(heap.begin(), heap.end(), above);
        }
    }
    out->core_off.assign(C + 1, 0);
    for (int32_t c = 0; c < C; ++c) out->core_off[c + 1] = out->core_off[c] + len[c];
    out->units.resize(nu);
    for (int32_t i = 0; i < nu; ++i) out->units[out->core_off[core_of[i]] + pos[i]] = u[i];
    out->makespan = nu ? *std::max_element(load.begin(), load.end()) : 0;
}

// ------------------------------------------------------- fused combine ----

constexpr int kCombineThreads = 256;  // 8 warps; one warp per (token, 256 elements)
constexpr int kRowBits = 40;          // a recorded copy row: owner * 2^40 + row
constexpr int kCombineSeg = 256;      // 32 lanes x 8 bf16 (16 bytes a lane)

struct RecvTable {
    const uint16_t* ex[MOE_EP_MAX_RANKS];  // each owner's bf16 receive rows
    int64_t rows[MOE_EP_MAX_RANKS];
};

// Lane j < k of a warp holds copy j of token t: its gate and its row's
// address in its owner's buffer -- the row the rank's fused dispatch recorded
// (RECORDED, one load), or recv_start[p] + slot - offsets[p] with p the
// copy's physical expert (two dependent loads more).  KB copies' 16-byte
// loads are in flight per lane before they are accumulated in ascending j,
// as in the single-GPU combine.
template <int KB, bool RECORDED>
__global__ void __launch_bounds__(kCombineThreads)
ep_combine_kernel(const int32_t* __restrict__ slot, const float* __restrict__ gates,
                  const int32_t* __restrict__ phys, const int32_t* __restrict__ offsets,
                  const int32_t* __restrict__ recv_start, const int64_t* __restrict__ copy_row, int T, int H, int k,
                  int R, int P, const RecvTable tab, uint16_t* __restrict__ y, int32_t* __restrict__ err) {
    grid_dependency_sync();
    const int lane = threadIdx.x & 31;
    const int segs = (H + kCombineSeg - 1) / kCombineSeg;
    const long long item = (long long)blockIdx.x * (kCombineThreads / 32) + (threadIdx.x >> 5);
    const int t = (int)(item / segs);
    const int seg = (int)(item - (long long)t * segs);
    if (t >= T) return;

    unsigned long long src = 0;  // address of this lane's copy's row
    float g = 0.0f;
    bool bad = false;
    if (lane < k) {
        g = gates[(size_t)t * k + lane];
        int d = -1;
        long long row = -1;
        if (RECORDED) {  // recorded by the fused dispatch: one load
            const long long v = copy_row[(size_t)t * k + lane];
            if (v >= 0) {
                d = (int)(v >> kRowBits);
                row = v & ((1LL << kRowBits) - 1);
            }
        } else {
            const int r = slot[(size_t)t * k + lane];
            const int p = phys[(size_t)t * k + lane];
            if (p >= 0 && p < P) {
                d = (int)(((long long)p * R) / P);
                row = (long long)recv_start[p] + r - offsets[p];
            }
        }
        if (d < 0 || d >= R || row < 0 || row >= tab.rows[d] || tab.ex[d] == nullptr)
            bad = true;
        else
            src = reinterpret_cast<unsigned long long>(tab.ex[d] + row * H);
    }
    if (__any_sync(kFull, bad)) {  // warp-uniform: skip the token's segment
        if (lane == 0) set_error(err, MOE_DEVERR_UNIT);
        return;
    }
    const int col = (seg * 32 + lane) * 8;
    const bool act = col < H;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
    for (int jb = 0; jb < k; jb += KB) {
        uint4 d[KB];
#pragma unroll
        for (int jj = 0; jj < KB; ++jj) {
            const int j = jb + jj;
            const unsigned long long a = __shfl_sync(kFull, src, j & 31);
            d[jj] = make_uint4(0, 0, 0, 0);
            if (j < k && act) d[jj] = ld_stream16(reinterpret_cast<const uint16_t*>(a) + col);
        }
#pragma unroll
        for (int jj = 0; jj < KB; ++jj) {
            const int j = jb + jj;
            const float gj = __shfl_sync(kFull, g, j & 31);
            if (j < k) {
                const uint32_t w[4] = {d[jj].x, d[jj].y, d[jj].z, d[jj].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    acc[2 * i] = __fmaf_rn(gj, bf16_lo(w[i]), acc[2 * i]);
                    acc[2 * i + 1] = __fmaf_rn(gj, bf16_hi(w[i]), acc[2 * i + 1]);
                }
            }
        }
    }
    if (act) {
        uint4 o;
        o.x = pack_bf16x2_rn(acc[0], acc[1]);
        o.y = pack_bf16x2_rn(acc[2], acc[3]);
        o.z = pack_bf16x2_rn(acc[4], acc[5]);
        o.w = pack_bf16x2_rn(acc[6], acc[7]);
        st16(y + (size_t)t * H + col, o);
    }
}

// ------------------------------------------------ window starts, device ----

constexpr int kStartThreads = 1024;

struct CountsTable {
    const int32_t* c[MOE_EP_MAX_RANKS];  // rank q's counts [P]
};

// One CTA: per expert the rows of all ranks (tot), their exclusive scan over
// the experts, each expert's window start inside its owner's buffer (the scan
// minus the scan at the owner's first expert), then each source's start
// inside the window (the counts of the ranks before it added up).
__global__ void __launch_bounds__(kStartThreads)
ep_recv_start_kernel(const CountsTable tab, int R, int P, int32_t* __restrict__ recv_start,
                     int32_t* __restrict__ recv_rows) {
    extern __shared__ long long excl[];  // [P + 1]
    __shared__ long long warp_tot[kStartThreads / 32];
    grid_dependency_sync();
    allow_dependents();
    const int per = (P + kStartThreads - 1) / kStartThreads;
    const int lo = threadIdx.x * per;
    long long chunk = 0;
    for (int p = lo; p < lo + per && p < P; ++p) {
        long long tot = 0;
        for (int q = 0; q < R; ++q) tot += tab.c[q][p];
        excl[p] = tot;
        chunk += tot;
    }
    // exclusive scan of the chunk totals over the CTA
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long incl = chunk;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    long long wsum = lane < kStartThreads / 32 ? warp_tot[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const long long o = __shfl_up_sync(kFull, wsum, off);
        if (lane >= off) wsum += o;
    }
    long long run = __shfl_sync(kFull, wsum, warp) - warp_tot[warp] + incl - chunk;
    __syncthreads();
    for (int p = lo; p < lo + per && p < P; ++p) {
        const long long v = excl[p];
        excl[p] = run;
        run += v;
    }
    if (threadIdx.x == kStartThreads - 1) excl[P] = run;
    __syncthreads();
    for (int p = threadIdx.x; p < P; p += kStartThreads) {
        const int d = (int)(((long long)p * R) / P);
        const int first = (int)(((long long)d * P + R - 1) / R);
        long long row = excl[p] - excl[first];
        for (int s = 0; s < R; ++s) {
            recv_start[(size_t)s * P + p] = (int32_t)row;
            row += tab.c[s][p];
        }
    }
    if (recv_rows != nullptr)
        for (int d = threadIdx.x; d < R; d += kStartThreads) {
            const int first = (int)(((long long)d * P + R - 1) / R);
            const int last = (int)(((long long)(d + 1) * P + R - 1) / R);
            recv_rows[d] = (int32_t)(excl[last] - excl[first]);
        }
}

// ---------------------------------------------------------- fused dispatch ----

constexpr int kDispatchThreads = 256;  // 8 warps, one per (token, 512-element segment)

struct SendTable {
    int8_t* codes[MOE_EP_MAX_RANKS];  // each owner's receive rows
    float* scales[MOE_EP_MAX_RANKS];
    int64_t rows[MOE_EP_MAX_RANKS];
};

// The dispatch of one rank written straight into the owners' receive
// buffers: per warp, one segment of one token is loaded and quantized once
// (quant.cuh), and lane j < k addresses copy j in its owner's buffer; the
// codes leave as one 16-byte store per lane and copy, the segment's four
// scales as one 16-byte store per copy.
__global__ void __launch_bounds__(kDispatchThreads)
ep_dispatch_kernel(const uint16_t* __restrict__ x, int T, int H, int k, int R, int P, int Gs,
                   const int32_t* __restrict__ slot, const int32_t* __restrict__ phys,
                   const int32_t* __restrict__ offsets, const int32_t* __restrict__ recv_start, const SendTable tab,
                   int64_t* __restrict__ copy_row, int32_t* __restrict__ err) {
    grid_dependency_sync();
    allow_dependents();
    const int lane = threadIdx.x & 31;
    const int segs = (H + kSegElems - 1) / kSegElems;
    const long long item = (long long)blockIdx.x * (kDispatchThreads / 32) + (threadIdx.x >> 5);
    const int t = (int)(item / segs);
    const int seg = (int)(item - (long long)t * segs);
    if (t >= T) return;
    const SegLoad ld = load_segment(x, t, H, seg, lane);
    unsigned long long cdst = 0;  // copy `lane`'s code row in its owner's buffer (0: skipped)
    float* sdst = nullptr;
    if (lane < k) {
        const int r = slot[(size_t)t * k + lane];
        const int p = phys[(size_t)t * k + lane];
        long long row = -1;
        int d = 0;
        if (p >= 0 && p < P) {
            d = (int)(((long long)p * R) / P);
            row = (long long)recv_start[p] + r - offsets[p];
        }
        const bool ok = row >= 0 && row < tab.rows[d] && tab.codes[d] != nullptr && tab.scales[d] != nullptr;
        if (!ok) {
            set_error(err, MOE_DEVERR_UNIT);
        } else {
            cdst = reinterpret_cast<unsigned long long>(tab.codes[d] + row * H);
            sdst = tab.scales[d] + row * Gs;
        }
        // where the copy went, once per copy (by the warp of segment 0)
        if (copy_row != nullptr && seg == 0)
            copy_row[(size_t)t * k + lane] = ok ? ((long long)d << kRowBits) | row : -1LL;
    }
    const SegQuant qz = quantize_segment(ld);
    for (int j = 0; j < k; ++j) {
        const unsigned long long a = __shfl_sync(kFull, cdst, j);
        if (a == 0) continue;  // warp-uniform
        if (ld.active) st16(reinterpret_cast<int8_t*>(a) + (size_t)ld.chunk * 16, qz.q);
    }
    if (sdst != nullptr && seg * 4 < Gs) *reinterpret_cast<float4*>(sdst + seg * 4) = qz.sc;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

MOE_API int moe_ep_experts(int32_t R, int32_t P, int32_t d, int32_t* first, int32_t* count) {
    if (first == nullptr || count == nullptr) return MOE_ERR_NULL;
    int rc = check_group(R, P);
    if (rc != MOE_OK) return rc;
    if (d < 0 || d >= R) return MOE_ERR_SIZE;
    *first = rank_first_expert(d, R, P);
    *count = rank_first_expert(d + 1, R, P) - *first;
    return MOE_OK;
}

MOE_API int moe_ep_layout(int32_t R, int32_t P, const int32_t* counts, int32_t d, int32_t* expert_off,
                          int32_t* chunk_row) {
    if (counts == nullptr || expert_off == nullptr || chunk_row == nullptr) return MOE_ERR_NULL;
    int32_t lo = 0, nd = 0;
    int rc = moe_ep_experts(R, P, d, &lo, &nd);
    if (rc != MOE_OK) return rc;
    int64_t row = 0;
    for (int32_t i = 0; i < nd; ++i) {
        expert_off[i] = (int32_t)row;
        for (int32_t s = 0; s < R; ++s) {
            chunk_row[(size_t)s * nd + i] = (int32_t)row;
            const int32_t n = counts[(size_t)s * P + lo + i];
            if (n < 0) return MOE_ERR_SIZE;
            row += n;
            if (row > INT32_MAX) return MOE_ERR_SIZE;
        }
    }
    expert_off[nd] = (int32_t)row;
    return MOE_OK;
}

MOE_API int moe_ep_max_units(const moe_ep_desc* desc, int64_t rows, int32_t* max_units) {
    if (max_units == nullptr) return MOE_ERR_NULL;
    int rc = check_desc(desc);
    if (rc != MOE_OK) return rc;
    if (rows < 0) return MOE_ERR_SIZE;
    const int64_t smin = std::min(desc->unit_rows[0], desc->unit_rows[1]);
    const int64_t nd_max = (desc->P + desc->R - 1) / desc->R;  // the largest block of experts
    const int64_t n = rows / smin + (int64_t)desc->R * nd_max;
    if (n > INT32_MAX) return MOE_ERR_SIZE;
    *max_units = (int32_t)n;
    return MOE_OK;
}

MOE_API int moe_ep_schedule(const moe_ep_desc* desc, int32_t direction, int32_t puller, const int32_t* counts,
                            int64_t row_bytes, moe_ep_unit* units, int32_t max_units, int32_t* n_units,
                            int32_t* core_off, int64_t* makespan_ps) {
    if (counts == nullptr || units == nullptr || n_units == nullptr || core_off == nullptr) return MOE_ERR_NULL;
    int rc = check_schedule_args(desc, direction, counts, row_bytes, max_units);
    if (rc != MOE_OK) return rc;
    if (puller < 0 || puller >= desc->R) return MOE_ERR_SIZE;
    Windows win;
    Schedule out;
    try {  // no exception leaves the C ABI: an allocation failure is a size error
        if ((rc = win.build(desc->R, desc->P, counts)) != MOE_OK) return rc;
        schedule_one(*desc, win, counts, direction, puller, row_bytes, &out);
    } catch (...) {
        return MOE_ERR_SIZE;
    }
    if ((int64_t)out.units.size() > max_units) return MOE_ERR_SIZE;
    std::copy(out.units.begin(), out.units.end(), units);
    std::copy(out.core_off.begin(), out.core_off.end(), core_off);
    *n_units = (int32_t)out.units.size();
    if (makespan_ps != nullptr) *makespan_ps = out.makespan;
    return MOE_OK;
}

MOE_API int moe_ep_schedule_group(const moe_ep_desc* desc, int32_t direction, const int32_t* counts,
                                  int64_t row_bytes, moe_ep_unit* units, int32_t max_units, int32_t* n_units,
                                  int32_t* core_off, int64_t* makespan_ps) {
    if (counts == nullptr || units == nullptr || n_units == nullptr || core_off == nullptr) return MOE_ERR_NULL;
    int rc = check_schedule_args(desc, direction, counts, row_bytes, max_units);
    if (rc != MOE_OK) return rc;
    const int32_t R = desc->R, C = desc->cores;
    Windows win;
    std::vector<Schedule> out;
    // One puller per task on the worker threads; each writes only its own
    // Schedule.  No exception leaves the C ABI: a failure in any task is a
    // size error.
    std::atomic<bool> failed{false};
    try {
        if ((rc = win.build(R, desc->P, counts)) != MOE_OK) return rc;
        out.resize((size_t)R);
        Workers::get().run(R, [&](int r) {
            try {
                schedule_one(*desc, win, counts, direction, r, row_bytes, &out[r]);
            } catch (...) {
                failed = true;
            }
        });
    } catch (...) {
        return MOE_ERR_SIZE;
    }
    if (failed) return MOE_ERR_SIZE;
    int64_t total = 0;
    for (const Schedule& sc : out) total += (int64_t)sc.units.size();
    if (total > max_units) return MOE_ERR_SIZE;
    int32_t base = 0;
    for (int32_t r = 0; r < R; ++r) {
        std::copy(out[r].units.begin(), out[r].units.end(), units + base);
        for (int32_t c = 0; c <= C; ++c) core_off[(size_t)r * (C + 1) + c] = base + out[r].core_off[c];
        if (makespan_ps != nullptr) makespan_ps[r] = out[r].makespan;
        base += (int32_t)out[r].units.size();
    }
    *n_units = base;
    return MOE_OK;
}

MOE_API int moe_ep_pull(const moe_ep_unit* units, const int32_t* core_off, int32_t n_units, int32_t R,
                        int32_t cores, int32_t first_puller, int32_t n_pullers, const moe_ep_plane* planes,
                        int32_t n_planes, int32_t* error_word, void* stream) {
    if (core_off == nullptr || planes == nullptr || error_word == nullptr) return MOE_ERR_NULL;
    if (units == nullptr && n_units > 0) return MOE_ERR_NULL;
    if (R < 1 || R > MOE_EP_MAX_RANKS || cores < 1 || cores > 4096 || n_pullers < 1 || first_puller < 0 ||
        first_puller + n_pullers > R || n_planes < 1 || n_planes > 2 || n_units < 0)
        return MOE_ERR_SIZE;
    auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (misaligned(units) || misaligned(error_word)) return MOE_ERR_ALIGN;
    PullPlanes pl;
    std::memset(&pl, 0, sizeof(pl));
    pl.n_planes = n_planes;
    for (int p = 0; p < n_planes; ++p) {
        const moe_ep_plane& a = planes[p];
        if (a.row_bytes < 16 || a.row_bytes % 16 != 0) return MOE_ERR_SIZE;
        pl.row_bytes[p] = a.row_bytes;
        for (int q = 0; q < R; ++q) {
            if (a.src_rows[q] < 0 || a.dst_rows[q] < 0) return MOE_ERR_SIZE;
            if (misaligned(a.src[q]) || misaligned(a.dst[q])) return MOE_ERR_ALIGN;
            pl.src[p][q] = static_cast<const char*>(a.src[q]);
            pl.dst[p][q] = static_cast<char*>(a.dst[q]);
            pl.src_rows[p][q] = a.src[q] == nullptr ? 0 : a.src_rows[q];
            pl.dst_rows[p][q] = a.dst[q] == nullptr ? 0 : a.dst_rows[q];
        }
    }
    cudaError_t e = launch_pdl(ep_pull_kernel, dim3((unsigned)cores, (unsigned)n_pullers), dim3(kPullThreads), 0,
                               static_cast<cudaStream_t>(stream), units, core_off, n_units, R, cores,
                               first_puller, pl, error_word);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

MOE_API int moe_ep_recv_start(int32_t R, int32_t P, const int32_t* counts, int32_t s, int32_t* recv_start) {
    if (counts == nullptr || recv_start == nullptr) return MOE_ERR_NULL;
    int rc = check_group(R, P);
    if (rc != MOE_OK) return rc;
    if (s < 0 || s >= R) return MOE_ERR_SIZE;
    for (int32_t d = 0; d < R; ++d) {
        int64_t row = 0;  // running row of d's receive buffer
        for (int32_t p = rank_first_expert(d, R, P); p < rank_first_expert(d + 1, R, P); ++p)
            for (int32_t q = 0; q < R; ++q) {
                const int32_t n = counts[(size_t)q * P + p];
                if (n < 0) return MOE_ERR_SIZE;
                if (q == s) recv_start[p] = (int32_t)row;
                row += n;
                if (row > INT32_MAX) return MOE_ERR_SIZE;
            }
    }
    return MOE_OK;
}

MOE_API int moe_ep_recv_start_device(int32_t R, int32_t P, const int32_t* const* counts, int32_t* recv_start,
                                     int32_t* recv_rows, void* stream) {
    if (counts == nullptr || recv_start == nullptr) return MOE_ERR_NULL;
    int rc = check_group(R, P);
    if (rc != MOE_OK) return rc;
    if ((reinterpret_cast<uintptr_t>(recv_start) & 3u) != 0 || (reinterpret_cast<uintptr_t>(recv_rows) & 3u) != 0)
        return MOE_ERR_ALIGN;
    CountsTable tab;
    std::memset(&tab, 0, sizeof(tab));
    for (int q = 0; q < R; ++q) {
        if (counts[q] == nullptr) return MOE_ERR_NULL;
        tab.c[q] = counts[q];
    }
    const size_t smem = (size_t)(P + 1) * sizeof(long long);
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024)
        e = cudaFuncSetAttribute(ep_recv_start_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
        e = launch_pdl(ep_recv_start_kernel, dim3(1), dim3(kStartThreads), smem, static_cast<cudaStream_t>(stream),
                       tab, R, P, recv_start, recv_rows);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

MOE_API int moe_ep_dispatch(moe_pool* pool, const uint16_t* x, int32_t T, int buf, int32_t R,
                            int8_t* const* recv_codes, float* const* recv_scales, const int64_t* recv_rows,
                            const int32_t* recv_start, int64_t* copy_row, void* stream) {
    if (pool == nullptr || recv_codes == nullptr || recv_scales == nullptr || recv_rows == nullptr)
        return MOE_ERR_NULL;
    const moe_desc& d = pool->geo.d;
    if (buf < 0 || buf >= d.n_sets) return MOE_ERR_BUF;
    if (T < 0 || T > d.T_max || R < 1 || R > MOE_EP_MAX_RANKS) return MOE_ERR_SIZE;
    if (pool->planned_T[buf] != T) return MOE_ERR_STATE;
    if (T == 0) return MOE_OK;
    if (x == nullptr || recv_start == nullptr) return MOE_ERR_NULL;
    auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (misaligned(x) || (reinterpret_cast<uintptr_t>(recv_start) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(copy_row) & 7u) != 0)
        return MOE_ERR_ALIGN;
    SendTable tab;
    std::memset(&tab, 0, sizeof(tab));
    for (int q = 0; q < R; ++q) {
        if (recv_rows[q] < 0) return MOE_ERR_SIZE;
        if (misaligned(recv_codes[q]) || misaligned(recv_scales[q])) return MOE_ERR_ALIGN;
        tab.codes[q] = recv_codes[q];
        tab.scales[q] = recv_scales[q];
        tab.rows[q] = (recv_codes[q] == nullptr || recv_scales[q] == nullptr) ? 0 : recv_rows[q];
        if (tab.rows[q] >= (1LL << kRowBits)) return MOE_ERR_SIZE;
    }
    const SetLayout& L = pool->geo.set[buf];
    char* base = pool->base;
    const long long items = (long long)T * ((d.H + kSegElems - 1) / kSegElems);
    const dim3 grid((unsigned)((items + (kDispatchThreads / 32) - 1) / (kDispatchThreads / 32)));
    cudaError_t e = launch_pdl(ep_dispatch_kernel, grid, dim3(kDispatchThreads), 0, static_cast<cudaStream_t>(stream),
                               x, T, d.H, d.k, R, d.P, pool->geo.Gs, reinterpret_cast<const int32_t*>(base + L.slot),
                               reinterpret_cast<const int32_t*>(base + L.phys),
                               reinterpret_cast<const int32_t*>(base + L.offsets), recv_start, tab, copy_row,
                               reinterpret_cast<int32_t*>(base + pool->geo.error_word));
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    pool->launches += 1;
    return MOE_OK;
}

MOE_API int moe_ep_combine(moe_pool* pool, int32_t T, int buf, int32_t R, const uint16_t* const* recv_ex,
                           const int64_t* recv_rows, const int32_t* recv_start, const int64_t* copy_row,
                           uint16_t* y, void* stream) {
    if (pool == nullptr || recv_ex == nullptr || recv_rows == nullptr) return MOE_ERR_NULL;
    const moe_desc& d = pool->geo.d;
    if (buf < 0 || buf >= d.n_sets) return MOE_ERR_BUF;
    if (T < 0 || T > d.T_max || R < 1 || R > MOE_EP_MAX_RANKS) return MOE_ERR_SIZE;
    if (pool->planned_T[buf] != T) return MOE_ERR_STATE;
    if (T == 0) return MOE_OK;
    if ((recv_start == nullptr && copy_row == nullptr) || y == nullptr) return MOE_ERR_NULL;
    auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if ((reinterpret_cast<uintptr_t>(recv_start) & 3u) != 0 || (reinterpret_cast<uintptr_t>(copy_row) & 7u) != 0 ||
        misaligned(y))
        return MOE_ERR_ALIGN;
    RecvTable tab;
    std::memset(&tab, 0, sizeof(tab));
    for (int q = 0; q < R; ++q) {
        if (recv_rows[q] < 0) return MOE_ERR_SIZE;
        if (misaligned(recv_ex[q])) return MOE_ERR_ALIGN;
        tab.ex[q] = recv_ex[q];
        tab.rows[q] = recv_ex[q] == nullptr ? 0 : recv_rows[q];
    }
    const SetLayout& L = pool->geo.set[buf];
    char* base = pool->base;
    const int32_t* slot = reinterpret_cast<const int32_t*>(base + L.slot);
    const float* gates = reinterpret_cast<const float*>(base + L.gates);
    const int32_t* phys = reinterpret_cast<const int32_t*>(base + L.phys);
    const int32_t* offsets = reinterpret_cast<const int32_t*>(base + L.offsets);
    int32_t* err = reinterpret_cast<int32_t*>(base + pool->geo.error_word);
    const long long items = (long long)T * ((d.H + kCombineSeg - 1) / kCombineSeg);
    const dim3 grid((unsigned)((items + (kCombineThreads / 32) - 1) / (kCombineThreads / 32)));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
#define MOE_EP_COMBINE_CASE(KB)                                                                              \
    e = copy_row != nullptr                                                                                   \
            ? launch_pdl(ep_combine_kernel<KB, true>, grid, dim3(kCombineThreads), 0, s, slot, gates, phys,   \
                         offsets, recv_start, copy_row, T, d.H, d.k, R, d.P, tab, y, err)                     \
            : launch_pdl(ep_combine_kernel<KB, false>, grid, dim3(kCombineThreads), 0, s, slot, gates, phys,  \
                         offsets, recv_start, copy_row, T, d.H, d.k, R, d.P, tab, y, err)
    switch (d.k < 8 ? d.k : 8) {
        case 1: MOE_EP_COMBINE_CASE(1); break;
        case 2: MOE_EP_COMBINE_CASE(2); break;
        case 3: MOE_EP_COMBINE_CASE(3); break;
        case 4: MOE_EP_COMBINE_CASE(4); break;
        case 5: MOE_EP_COMBINE_CASE(5); break;
        case 6: MOE_EP_COMBINE_CASE(6); break;
        case 7: MOE_EP_COMBINE_CASE(7); break;
        default: MOE_EP_COMBINE_CASE(8); break;
    }
#undef MOE_EP_COMBINE_CASE
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    pool->launches += 1;
    return MOE_OK;
}

MOE_API int moe_dequant_rows(const int8_t* codes, const float* scales, int32_t rows, int32_t H,
                             int32_t scale_stride, uint16_t* out, void* stream) {
    if (rows < 0 || H < kGroup || H > 65536 || H % kGroup != 0 || scale_stride < H / kGroup ||
        scale_stride % 4 != 0)
        return MOE_ERR_SIZE;
    if (rows == 0) return MOE_OK;
    if (codes == nullptr || scales == nullptr || out == nullptr) return MOE_ERR_NULL;
    auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
    if (misaligned(codes) || misaligned(scales) || misaligned(out)) return MOE_ERR_ALIGN;
    uint64_t launches = 0;
    cudaError_t e = launch_identity_experts(codes, scales, rows, H, scale_stride, out,
                                            static_cast<cudaStream_t>(stream), &launches);
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
