/*
 * moe_trace.h -- stage probes of the libmoe kernels (trace build only).
 *
 * Exported only by libmoe_trace.so, the same library compiled with
 * -DMOE_TRACE; libmoe.so exports none of these.  It follows the NPU-side
 * profiler of the StrataCL analysis (section 3.7): inline probes at the phase
 * boundaries of each kernel, stamped with an on-chip clock into a per-core
 * trace slice that the host decodes into per-core timelines.
 *
 * For every kernel kind below, thread 0 of each of the first MOE_TRACE_CTAS
 * CTAs records, at each stage boundary s < MOE_TRACE_STAGES, the pair
 * (%globaltimer in ns, clock64 in SM cycles), and once the id of the SM it ran
 * on.  Stage meanings are listed per kind.  A stamp of 0 means "not reached"
 * (a CTA that exited early, or a stage its kernel does not have).  Each launch
 * of a kind overwrites that kind's stamps: read them after the launch you
 * want and before the next one of the same kind.
 */
#ifndef MOE_TRACE_H
#define MOE_TRACE_H

#include <stddef.h>
#include <stdint.h>

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_TRACE_CTAS 8192
#define MOE_TRACE_STAGES 12

typedef enum moe_trace_kind {
    MOE_TRACE_ROUTE = 0,       /* route_tile: 0 start, 1 top-k, 2 exp, 3 sums, 4 gates+masks, 5 counts+ranks */
    MOE_TRACE_COLUMN_SCAN = 1, /* column_scan: 0 start, 1 end */
    MOE_TRACE_ASSIGN = 2,      /* assign: 0 start, 1 offsets, 2 end */
    MOE_TRACE_PLAN_SINGLE = 3, /* one-launch plan, 0-5 as route: the cluster kernel (6 cluster
                                  barrier passed, 7 other tiles' masks read, 8 offsets
                                  scanned, 9 copies placed) or, without clusters, the ticket
                                  kernel (last CTA: 6 tail start, 7 end) */
    MOE_TRACE_DISPATCH = 4,    /* dispatch (warp 0): 0 start, 1 quantized, 2 slots read, 3 stored */
    MOE_TRACE_COMBINE = 5,     /* combine (warp 0): 0 start, 1 slots, 2 accumulated, 3 stored */
    MOE_TRACE_KINDS = 6
} moe_trace_kind;

/* Zero every kind's stamps and SM ids (asynchronous on `stream`). */
MOE_API int moe_trace_reset(void* stream);

/*
 * Synchronous copy of one kind's records to the host.
 *   stamps  uint64 [MOE_TRACE_CTAS][MOE_TRACE_STAGES][2] (ns, cycles), or NULL
 *   sm_ids  uint32 [MOE_TRACE_CTAS], or NULL
 * Returns MOE_ERR_SIZE for an unknown kind, MOE_ERR_CUDA if a copy fails.
 */
MOE_API int moe_trace_read(int kind, uint64_t* stamps, uint32_t* sm_ids);

#ifdef __cplusplus
}
#endif

#endif /* MOE_TRACE_H */
