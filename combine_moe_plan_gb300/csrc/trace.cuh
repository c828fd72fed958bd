// trace.cuh -- in-kernel stage probes (trace build only).
//
// StrataCL analysis, section 3.7 (NPU-side profiler): inline probes at the
// phase boundaries of a communication kernel, stamped with an on-chip clock
// into a per-core slice of a trace buffer, decoded on the host into per-core
// timelines.  Here: thread 0 of every CTA stamps %globaltimer (ns, common to
// all SMs), clock64 (SM cycles) and %smid at each stage boundary of the
// kernel into a per-kernel array [CTA][stage].  Compiled in only with
// -DMOE_TRACE (libmoe_trace.so); in the product build every probe is empty.
#pragma once

#include <cstdint>

namespace moe {

constexpr int kTraceCtas = 8192;  // CTAs recorded per kernel (later CTAs are not)
constexpr int kTraceStages = 12;  // stage stamps per CTA

// Trace slots: one per kernel kind.
enum TraceKind : int {
    kTraceRoute = 0,
    kTraceColumnScan = 1,
    kTraceAssign = 2,
    kTracePlanSingle = 3,
    kTraceDispatch = 4,
    kTraceCombine = 5,
    kTraceKinds = 6
};

struct TraceStamp {
    unsigned long long ns;      // %globaltimer
    unsigned long long cycles;  // clock64 of the CTA's SM
};

#ifdef MOE_TRACE
using TraceSlice = TraceStamp (*)[kTraceStages];

__device__ __forceinline__ void trace_mark(TraceSlice buf, int stage) {
    if (threadIdx.x == 0 && blockIdx.x < (unsigned)kTraceCtas) {
        unsigned long long g;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(g));
        buf[blockIdx.x][stage].ns = g;
        buf[blockIdx.x][stage].cycles = (unsigned long long)clock64();
    }
}
__device__ __forceinline__ void trace_sm(unsigned* sm_buf) {
    if (threadIdx.x == 0 && blockIdx.x < (unsigned)kTraceCtas) {
        unsigned id;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(id));
        sm_buf[blockIdx.x] = id;
    }
}
// Each kernel file declares its own buffers (no cross-file device symbols):
//   MOE_TRACE_BUFFERS(name) -> static __device__ arrays name##_t / name##_sm
#define MOE_TRACE_BUFFERS(name)                                                \
    static __device__ moe::TraceStamp name##_t[moe::kTraceCtas][moe::kTraceStages]; \
    static __device__ unsigned name##_sm[moe::kTraceCtas];
#define MOE_TRACE_MARK(name, stage) moe::trace_mark(name##_t, (stage))
#define MOE_TRACE_SM(name) moe::trace_sm(name##_sm)
#else
#define MOE_TRACE_BUFFERS(name)
#define MOE_TRACE_MARK(name, stage) ((void)0)
#define MOE_TRACE_SM(name) ((void)0)
#endif

// Host side (trace build): device addresses of a kind's buffers, looked up
// with cudaGetSymbolAddress in the file that owns them.
int trace_symbols_plan(int kind, void** stamps, void** sms);
int trace_symbols_dispatch(void** stamps, void** sms);
int trace_symbols_combine(void** stamps, void** sms);

}  // namespace moe
