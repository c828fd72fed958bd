// trace.cu -- host side of the stage probes (trace build only; empty otherwise).
#ifdef MOE_TRACE
#include "moe_trace.h"

#include "moe_internal.h"
#include "trace.cuh"

namespace {

int symbols(int kind, void** stamps, void** sms) {
    switch (kind) {
        case MOE_TRACE_ROUTE:
        case MOE_TRACE_COLUMN_SCAN:
        case MOE_TRACE_ASSIGN:
        case MOE_TRACE_PLAN_SINGLE:
            return moe::trace_symbols_plan(kind, stamps, sms);
        case MOE_TRACE_DISPATCH:
            return moe::trace_symbols_dispatch(stamps, sms);
        case MOE_TRACE_COMBINE:
            return moe::trace_symbols_combine(stamps, sms);
        default:
            return -1;
    }
}

constexpr size_t kStampBytes = sizeof(moe::TraceStamp) * moe::kTraceCtas * moe::kTraceStages;
constexpr size_t kSmBytes = sizeof(unsigned) * moe::kTraceCtas;

}  // namespace

extern "C" MOE_API int moe_trace_reset(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    for (int kind = 0; kind < MOE_TRACE_KINDS; ++kind) {
        void *st = nullptr, *sm = nullptr;
        if (symbols(kind, &st, &sm) != 0) return MOE_ERR_CUDA;
        if (cudaMemsetAsync(st, 0, kStampBytes, s) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaMemsetAsync(sm, 0, kSmBytes, s) != cudaSuccess) return MOE_ERR_CUDA;
    }
    return MOE_OK;
}

extern "C" MOE_API int moe_trace_read(int kind, uint64_t* stamps, uint32_t* sm_ids) {
    if (kind < 0 || kind >= MOE_TRACE_KINDS) return MOE_ERR_SIZE;
    void *st = nullptr, *sm = nullptr;
    if (symbols(kind, &st, &sm) != 0) return MOE_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
    if (stamps != nullptr && cudaMemcpy(stamps, st, kStampBytes, cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (sm_ids != nullptr && cudaMemcpy(sm_ids, sm, kSmBytes, cudaMemcpyDeviceToHost) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
#endif
