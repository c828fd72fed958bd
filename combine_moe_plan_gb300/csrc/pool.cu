// pool.cu -- libmoe C ABI: static buffer pool, argument checks, launches.
//
// The pool is the GPU form of the write-up's "Double-Buffered Static
// Pre-allocation" (CloudMatrix384, "FusedDispatch and FusedCombine"):
// separate dispatch (INT8 codes + scales) and combine (bf16 expert outputs)
// buffers, sized once for the worst case, carved from one caller-owned
// workspace, with n_sets copies so consecutive iterations alternate sets.
// No call allocates; every launch is asynchronous on the caller's stream.
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <vector>

#include "moe_internal.h"

namespace moe {

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_desc(const moe_desc* d) {
    if (d == nullptr) return MOE_ERR_NULL;
    if (d->T_max < 1 || d->T_max > (1 << 20)) return MOE_ERR_SIZE;
    if (d->H < kGroup || d->H > 65536 || d->H % kGroup != 0) return MOE_ERR_SIZE;
    if (d->E < 1 || d->E > 1024) return MOE_ERR_SIZE;
    if (d->P < d->E || d->P > 4096) return MOE_ERR_SIZE;
    if (d->k < 1 || d->k > d->E || d->k > 32) return MOE_ERR_SIZE;
    if (d->group != kGroup) return MOE_ERR_SIZE;
    if (d->n_sets < 1 || d->n_sets > kMaxSets) return MOE_ERR_SIZE;
    if ((int64_t)d->T_max * d->k > (int64_t)INT32_MAX / 2) return MOE_ERR_SIZE;
    return MOE_OK;
}

}  // namespace

int make_geometry(const moe_desc* d, Geometry* g) {
    int rc = check_desc(d);
    if (rc != MOE_OK) return rc;
    std::memset(g, 0, sizeof(*g));
    g->d = *d;
    g->rows = (int64_t)d->T_max * d->k;
    g->G = d->H / kGroup;
    g->Gs = (g->G + 3) / 4 * 4;
    // route_tiles over T <= T_max: ceil(T / 32), or ceil(T / 16) up to 2048 tokens.
    g->tiles_max = std::max(route_tiles(d->T_max, d->E, d->k),
                            route_tiles(std::min(d->T_max, kMidTileMaxTokens), d->E, d->k));
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, kAlign);
        return o;
    };
    // Control block: error word, then one plan ticket per set.
    g->error_word = 0;
    g->ticket = 16;
    g->control_bytes = g->ticket + (size_t)d->n_sets * sizeof(int32_t);
    take(g->control_bytes);
    const size_t R = (size_t)g->rows, H = (size_t)d->H, T = (size_t)d->T_max, k = (size_t)d->k;
    for (int s = 0; s < d->n_sets; ++s) {
        SetLayout& L = g->set[s];
        L.codes = take(R * H);
        L.scales = take(R * (size_t)g->Gs * sizeof(float));
        L.ex_out = take(R * H * sizeof(uint16_t));
        L.topk_e = take(T * k * sizeof(int32_t));
        L.phys = take(T * k * sizeof(int32_t));
        L.gates = take(T * k * sizeof(float));
        L.slot = take(T * k * sizeof(int32_t));
        L.src_token = take(R * sizeof(int32_t));
        L.src_k = take(R * sizeof(int32_t));
        L.counts = take((size_t)d->P * sizeof(int32_t));
        L.offsets = take((size_t)(d->P + 1) * sizeof(int32_t));
        L.tile_hist = take((size_t)d->P * (size_t)g->tiles_max * sizeof(int32_t));
        L.local_rank = take(T * k * sizeof(int32_t));
        L.x_stage = take(T * H * sizeof(uint16_t));
        L.logits_stage = take(T * (size_t)d->E * sizeof(float));
        L.y_stage = take(T * H * sizeof(uint16_t));
    }
    g->total = off;
    return MOE_OK;
}

}  // namespace moe

using namespace moe;

namespace {

template <typename T>
T* at(const moe_pool* p, size_t off) {
    return reinterpret_cast<T*>(p->base + off);
}

int check_call(const moe_pool* pool, int32_t T, int buf) {
    if (pool == nullptr) return MOE_ERR_NULL;
    if (buf < 0 || buf >= pool->geo.d.n_sets) return MOE_ERR_BUF;
    if (T < 0 || T > pool->geo.d.T_max) return MOE_ERR_SIZE;
    return MOE_OK;
}

// The replica-map arguments of a non-empty plan: both pointers or neither
// (neither requires P == E), each 16-byte aligned.
int check_replica_args(const moe_desc& d, const int32_t* rep_off, const int32_t* rep_ids) {
    if ((rep_off == nullptr) != (rep_ids == nullptr)) return MOE_ERR_NULL;
    if (rep_off == nullptr && d.P != d.E) return MOE_ERR_REPLICA;
    if (rep_off != nullptr && (!aligned16(rep_off) || !aligned16(rep_ids))) return MOE_ERR_ALIGN;
    return MOE_OK;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

}  // namespace

extern "C" {

MOE_API int moe_pool_bytes(const moe_desc* desc, size_t* bytes) {
    if (bytes == nullptr) return MOE_ERR_NULL;
    Geometry g;
    int rc = make_geometry(desc, &g);
    if (rc != MOE_OK) return rc;
    *bytes = g.total;
    return MOE_OK;
}

MOE_API int moe_pool_init(const moe_desc* desc, void* dev_ws, size_t ws_bytes, moe_pool** out) {
    if (out == nullptr || dev_ws == nullptr) return MOE_ERR_NULL;
    *out = nullptr;
    Geometry g;
    int rc = make_geometry(desc, &g);
    if (rc != MOE_OK) return rc;
    if ((reinterpret_cast<uintptr_t>(dev_ws) & 255u) != 0) return MOE_ERR_ALIGN;
    if (ws_bytes < g.total) return MOE_ERR_WORKSPACE;
    moe_pool* p = static_cast<moe_pool*>(std::calloc(1, sizeof(moe_pool)));
    if (p == nullptr) return MOE_ERR_SIZE;
    p->geo = g;
    p->base = static_cast<char*>(dev_ws);
    for (int b = 0; b < kMaxSets; ++b) p->planned_T[b] = -1;
    *out = p;
    return MOE_OK;
}

MOE_API int moe_pool_destroy(moe_pool* pool) {
    if (pool == nullptr) return MOE_ERR_NULL;
    std::free(pool);
    return MOE_OK;
}

MOE_API int moe_pool_view(const moe_pool* pool, int buf, moe_view* v) {
    if (pool == nullptr || v == nullptr) return MOE_ERR_NULL;
    if (buf < 0 || buf >= pool->geo.d.n_sets) return MOE_ERR_BUF;
    const SetLayout& L = pool->geo.set[buf];
    v->codes = at<int8_t>(pool, L.codes);
    v->scales = at<float>(pool, L.scales);
    v->ex_out = at<uint16_t>(pool, L.ex_out);
    v->topk_e = at<int32_t>(pool, L.topk_e);
    v->phys = at<int32_t>(pool, L.phys);
    v->gates = at<float>(pool, L.gates);
    v->slot = at<int32_t>(pool, L.slot);
    v->src_token = at<int32_t>(pool, L.src_token);
    v->src_k = at<int32_t>(pool, L.src_k);
    v->counts = at<int32_t>(pool, L.counts);
    v->offsets = at<int32_t>(pool, L.offsets);
    v->error_word = at<int32_t>(pool, pool->geo.error_word);
    v->rows = (int32_t)pool->geo.rows;
    v->scale_stride = pool->geo.Gs;
    return MOE_OK;
}

MOE_API int moe_pool_clear_error(moe_pool* pool, void* stream) {
    if (pool == nullptr) return MOE_ERR_NULL;
    return cuda_rc(cudaMemsetAsync(pool->base, 0, pool->geo.control_bytes, static_cast<cudaStream_t>(stream)));
}

MOE_API int moe_pool_check(moe_pool* pool, void* stream, int32_t* error_word) {
    if (pool == nullptr) return MOE_ERR_NULL;
    int32_t w = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&w, at<int32_t>(pool, pool->geo.error_word), sizeof(w),
                                    cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    if (error_word != nullptr) *error_word = w;
    return w ? MOE_ERR_DEVICE : MOE_OK;
}

MOE_API int moe_pool_launches(const moe_pool* pool, uint64_t* count) {
    if (pool == nullptr || count == nullptr) return MOE_ERR_NULL;
    *count = pool->launches;
    return MOE_OK;
}

MOE_API int moe_replica_check(const int32_t* rep_off, const int32_t* rep_ids, int32_t E, int32_t P) {
    if (rep_off == nullptr || rep_ids == nullptr) return MOE_ERR_NULL;
    if (E < 1 || P < E) return MOE_ERR_SIZE;
    if (rep_off[0] != 0 || rep_off[E] != P) return MOE_ERR_REPLICA;
    for (int32_t e = 0; e < E; ++e)
        if (rep_off[e + 1] - rep_off[e] < 1) return MOE_ERR_REPLICA;
    std::vector<char> seen((size_t)P, 0);
    for (int32_t i = 0; i < P; ++i) {
        const int32_t p = rep_ids[i];
        if (p < 0 || p >= P || seen[(size_t)p]) return MOE_ERR_REPLICA;
        seen[(size_t)p] = 1;
    }
    return MOE_OK;
}

MOE_API int moe_plan(moe_pool* pool, const float* logits, int32_t T, const int32_t* rep_off,
                     const int32_t* rep_ids, int buf, void* stream) {
    int rc = check_call(pool, T, buf);
    if (rc != MOE_OK) return rc;
    const moe_desc& d = pool->geo.d;
    const SetLayout& L = pool->geo.set[buf];
    pool->planned_T[buf] = -1;
    if (T == 0) {  // an empty batch: every expert window is empty
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        if (cudaMemsetAsync(at<int32_t>(pool, L.counts), 0, (size_t)d.P * sizeof(int32_t), s) != cudaSuccess ||
            cudaMemsetAsync(at<int32_t>(pool, L.offsets), 0, (size_t)(d.P + 1) * sizeof(int32_t), s) !=
                cudaSuccess)
            return MOE_ERR_CUDA;
        pool->planned_T[buf] = 0;
        return MOE_OK;
    }
    if (logits == nullptr) return MOE_ERR_NULL;
    if (!aligned16(logits)) return MOE_ERR_ALIGN;
    if ((rc = check_replica_args(d, rep_off, rep_ids)) != MOE_OK) return rc;
    cudaError_t e = launch_plan(logits, T, d.E, d.P, d.k, rep_off, rep_ids, at<int32_t>(pool, L.topk_e),
                                at<float>(pool, L.gates), at<int32_t>(pool, L.phys),
                                at<int32_t>(pool, L.tile_hist), at<int32_t>(pool, L.local_rank),
                                at<int32_t>(pool, L.counts), at<int32_t>(pool, L.offsets),
                                at<int32_t>(pool, L.slot), at<int32_t>(pool, L.src_token),
                                at<int32_t>(pool, L.src_k), at<int32_t>(pool, pool->geo.error_word),
                                at<int32_t>(pool, pool->geo.ticket) + buf, static_cast<cudaStream_t>(stream),
                                &pool->launches);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    pool->planned_T[buf] = T;
    return MOE_OK;
}

}  // extern "C"

namespace {

int dispatch_call(moe_pool* pool, const uint16_t* x, int32_t T, int buf, bool x_early, void* stream) {
    int rc = check_call(pool, T, buf);
    if (rc != MOE_OK) return rc;
    if (T > 0 && x == nullptr) return MOE_ERR_NULL;
    if (T > 0 && !aligned16(x)) return MOE_ERR_ALIGN;
    if (pool->planned_T[buf] != T) return MOE_ERR_STATE;
    if (T == 0) return MOE_OK;
    const moe_desc& d = pool->geo.d;
    const SetLayout& L = pool->geo.set[buf];
    return cuda_rc(launch_dispatch(x, T, d.H, d.k, at<int32_t>(pool, L.slot), at<int8_t>(pool, L.codes),
                                   at<float>(pool, L.scales), pool->geo.Gs,
                                   at<int32_t>(pool, pool->geo.error_word), x_early,
                                   static_cast<cudaStream_t>(stream), &pool->launches));
}

}  // namespace

extern "C" {

MOE_API int moe_dispatch(moe_pool* pool, const uint16_t* x, int32_t T, int buf, void* stream) {
    return dispatch_call(pool, x, T, buf, false, stream);
}

MOE_API int moe_dispatch_after_plan(moe_pool* pool, const uint16_t* x, int32_t T, int buf, void* stream) {
    return dispatch_call(pool, x, T, buf, true, stream);
}

MOE_API int moe_plan_dispatch(moe_pool* pool, const float* logits, int32_t T, const int32_t* rep_off,
                              const int32_t* rep_ids, const uint16_t* x, int buf, void* stream) {
    int rc = check_call(pool, T, buf);
    if (rc != MOE_OK) return rc;
    if (T > 0 && x == nullptr) return MOE_ERR_NULL;
    if (T > 0 && !aligned16(x)) return MOE_ERR_ALIGN;
    // The plan checks the rest before launching; with x checked first, an
    // error leaves nothing enqueued.
    if ((rc = moe_plan(pool, logits, T, rep_off, rep_ids, buf, stream)) != MOE_OK) return rc;
    // The plan is the kernel just before, so the dispatch may load x while it
    // runs: x was written before the plan in stream order.
    return dispatch_call(pool, x, T, buf, true, stream);
}

MOE_API int moe_identity_experts(moe_pool* pool, int32_t T, int buf, void* stream) {
    int rc = check_call(pool, T, buf);
    if (rc != MOE_OK) return rc;
    if (pool->planned_T[buf] != T) return MOE_ERR_STATE;
    if (T == 0) return MOE_OK;
    const moe_desc& d = pool->geo.d;
    const SetLayout& L = pool->geo.set[buf];
    return cuda_rc(launch_identity_experts(at<int8_t>(pool, L.codes), at<float>(pool, L.scales), T * d.k, d.H,
                                           pool->geo.Gs, at<uint16_t>(pool, L.ex_out),
                                           static_cast<cudaStream_t>(stream), &pool->launches));
}

MOE_API int moe_combine(moe_pool* pool, const uint16_t* ex_out, uint16_t* y, int32_t T, int buf, void* stream) {
    int rc = check_call(pool, T, buf);
    if (rc != MOE_OK) return rc;
    if (T > 0 && y == nullptr) return MOE_ERR_NULL;
    if (T > 0 && (!aligned16(y) || (ex_out != nullptr && !aligned16(ex_out)))) return MOE_ERR_ALIGN;
    if (pool->planned_T[buf] != T) return MOE_ERR_STATE;
    if (T == 0) return MOE_OK;
    const moe_desc& d = pool->geo.d;
    const SetLayout& L = pool->geo.set[buf];
    const uint16_t* src = ex_out != nullptr ? ex_out : at<uint16_t>(pool, L.ex_out);
    return cuda_rc(launch_combine(src, at<int32_t>(pool, L.slot), at<float>(pool, L.gates), T, d.H, d.k, y,
                                  at<int32_t>(pool, pool->geo.error_word), static_cast<cudaStream_t>(stream),
                                  &pool->launches));
}

MOE_API int moe_step_host(moe_pool* pool, const float* h_logits, const uint16_t* h_x, const uint16_t* h_ex_out,
                          uint16_t* h_y, int32_t T, const int32_t* rep_off, const int32_t* rep_ids, int buf,
                          void* stream) {
    int rc = check_call(pool, T, buf);
    if (rc != MOE_OK) return rc;
    if (T == 0) return moe_plan(pool, h_logits, 0, rep_off, rep_ids, buf, stream);
    if (h_logits == nullptr || h_x == nullptr || h_y == nullptr) return MOE_ERR_NULL;
    const moe_desc& d = pool->geo.d;
    // Everything moe_plan would reject is rejected before the first copy, so
    // that on an error nothing is enqueued.
    if ((rc = check_replica_args(d, rep_off, rep_ids)) != MOE_OK) return rc;
    const SetLayout& L = pool->geo.set[buf];
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float* logits = at<float>(pool, L.logits_stage);
    uint16_t* x = at<uint16_t>(pool, L.x_stage);
    uint16_t* y = at<uint16_t>(pool, L.y_stage);
    const size_t TH = (size_t)T * d.H;
    if (cudaMemcpyAsync(logits, h_logits, (size_t)T * d.E * sizeof(float), cudaMemcpyHostToDevice, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(x, h_x, TH * sizeof(uint16_t), cudaMemcpyHostToDevice, s) != cudaSuccess)
        return MOE_ERR_CUDA;
    if ((rc = moe_plan_dispatch(pool, logits, T, rep_off, rep_ids, x, buf, stream)) != MOE_OK) return rc;
    if (h_ex_out != nullptr) {
        if (cudaMemcpyAsync(at<uint16_t>(pool, L.ex_out), h_ex_out, (size_t)T * d.k * d.H * sizeof(uint16_t),
                            cudaMemcpyHostToDevice, s) != cudaSuccess)
            return MOE_ERR_CUDA;
    } else if ((rc = moe_identity_experts(pool, T, buf, stream)) != MOE_OK) {
        return rc;
    }
    if ((rc = moe_combine(pool, nullptr, y, T, buf, stream)) != MOE_OK) return rc;
    return cuda_rc(cudaMemcpyAsync(h_y, y, TH * sizeof(uint16_t), cudaMemcpyDeviceToHost, s));
}

MOE_API const char* moe_status_str(int status) {
    switch (status) {
        case MOE_OK: return "ok";
        case MOE_ERR_NULL: return "required pointer is NULL";
        case MOE_ERR_SIZE: return "size out of range";
        case MOE_ERR_ALIGN: return "pointer not 16-byte aligned";
        case MOE_ERR_BUF: return "buffer set index out of range";
        case MOE_ERR_WORKSPACE: return "workspace smaller than moe_pool_bytes";
        case MOE_ERR_CUDA: return "CUDA runtime call failed";
        case MOE_ERR_DEVICE: return "kernel reported a bad index (device error word)";
        case MOE_ERR_REPLICA: return "malformed replica map";
        case MOE_ERR_STATE: return "T differs from the T planned for this buffer set";
        default: return "unknown status";
    }
}

}  // extern "C"
