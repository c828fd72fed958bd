/*
 * moe.h -- C ABI of libmoe: MoE FusedDispatch / FusedCombine on one GPU.
 *
 * The method (CloudMatrix384 write-up, section "FusedDispatch and
 * FusedCombine") replaces the three exchanges of an all-to-all MoE layer --
 * routing metadata, token data, expert output return -- with two fused
 * operators that write straight into statically pre-allocated, double-buffered
 * per-expert buffers, quantize tokens to INT8 before they move, and run a
 * token-granular load -> quantize/address -> write pipeline.  Here the
 * per-expert buffers are expert-major windows of one pool in local HBM.
 *
 * Calls, in the order one MoE layer uses them:
 *   moe_plan      routing metadata: top-k, gates, replica map, histogram,
 *                 exclusive scan, stable slot assignment ("metadata
 *                 generation and token reordering before dispatch",
 *                 write-up section "Prefill Phase"; expert-window aggregation,
 *                 StrataCL analysis section 3.5).
 *   moe_dispatch  fused per-token INT8 quantization (one fp32 scale per 128
 *                 elements) and scatter of each token into its k slots
 *                 (write-up: "Early INT8 Quantization", "AIV-Direct Write",
 *                 "Token-Level Pipeline").
 *   moe_plan_dispatch  both in one call; the dispatch then reads x while
 *                 the plan runs, safely.
 *   (experts)     outside this library; moe_identity_experts is a stand-in
 *                 that dequantizes each slot row (code * scale -> bf16).
 *   moe_combine   gate-weighted gather-reduce of the k bf16 expert rows back
 *                 to token order, fp32 fma in ascending j (write-up: "expert
 *                 output return").
 *
 * Conventions for every call:
 *   - Return 0 (MOE_OK) or a negative moe_status.  Arguments are checked on
 *     the host before anything is launched; on an error nothing is enqueued.
 *   - Device pointers are plain addresses in the current device's memory.
 *     Tensors are dense row-major.  bf16 values travel as uint16_t bit
 *     patterns.  Every device pointer must be 16-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  All
 *     work is asynchronous on that stream; nothing synchronizes except
 *     moe_pool_check and moe_step_host's documented copies.
 *   - Kernels are launched with programmatic dependent launch: each may start
 *     while the kernel before it on the stream drains, and waits for it
 *     (griddepcontrol.wait) before reading any input; each lets its own
 *     dependents start only after that wait.  So every input written earlier
 *     in stream order, by any kernel or copy, is seen.  The one opt-in
 *     exception is moe_dispatch_after_plan, which reads x before its wait
 *     (see there).
 *   - The caller owns every buffer, including the pool workspace; the library
 *     never allocates device memory.
 *   - Inputs outside the documented domain (non-finite logits or activations,
 *     |x| >= 2^120) give unspecified values but no out-of-bounds access.
 *   - Kernels check every index they compute from data (replica map, slots);
 *     a bad one skips the access and sets a bit in the pool's device error
 *     word, read by moe_pool_check.  No kernel traps or waits on a flag.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(_WIN32)
#define MOE_API
#else
#define MOE_API __attribute__((visibility("default")))
#endif

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_NULL = -1,      /* a required pointer is NULL */
    MOE_ERR_SIZE = -2,      /* a size is out of range (see moe_desc) */
    MOE_ERR_ALIGN = -3,     /* a pointer is not 16-byte aligned */
    MOE_ERR_BUF = -4,       /* buffer-set index outside [0, n_sets) */
    MOE_ERR_WORKSPACE = -5, /* workspace smaller than moe_pool_bytes */
    MOE_ERR_CUDA = -6,      /* a CUDA runtime call failed */
    MOE_ERR_DEVICE = -7,    /* a kernel reported a bad index (error word) */
    MOE_ERR_REPLICA = -8,   /* malformed replica map (host check) */
    MOE_ERR_STATE = -9      /* T differs from the one planned for this set */
} moe_status;

/* Device error-word bits (moe_pool_check). */
#define MOE_DEVERR_REPLICA 0x1   /* replica map gave an id outside [0, P) */
#define MOE_DEVERR_DUPLICATE 0x2 /* a token mapped twice to one physical expert */
#define MOE_DEVERR_SLOT 0x4      /* a slot index outside [0, T*k) */

/*
 * Pool geometry, fixed at init (static pre-allocation: write-up,
 * "Double-Buffered Static Pre-allocation").
 *   T_max   largest token count any call will use, 1 .. 2^20
 *   H       hidden size, a multiple of 128, 128 .. 65536
 *   E       logical experts, 1 .. 1024
 *   P       physical expert slots (E + redundant replicas), E .. 4096
 *   k       experts per token, 1 .. min(E, 32)
 *   group   quantization group, must be 128
 *   n_sets  buffer sets for double buffering, 1 .. 4 (2 = double buffered)
 * Worst-case capacity: every set holds T_max*k dispatched rows, so any
 * routing (up to all tokens on one expert) fits without dropping.
 */
typedef struct moe_desc {
    int32_t T_max, H, E, P, k, group, n_sets;
} moe_desc;

typedef struct moe_pool moe_pool; /* opaque host-side handle */

/*
 * Device addresses of one buffer set, carved from the workspace.  Sizes in
 * elements; R = T_max * k rows; Gs = H/128 rounded up to a multiple of 4.
 */
typedef struct moe_view {
    int8_t* codes;       /* [R, H] INT8 dispatch rows, expert-major windows */
    float* scales;       /* [R, Gs] fp32 scale per 128-element group (Gs-G pad) */
    uint16_t* ex_out;    /* [R, H] bf16 expert outputs (combine buffer) */
    int32_t* topk_e;     /* [T_max, k] logical expert per (t, j) */
    int32_t* phys;       /* [T_max, k] physical expert per (t, j) */
    float* gates;        /* [T_max, k] fp32 gate per (t, j) */
    int32_t* slot;       /* [T_max, k] row of copy (t, j) */
    int32_t* src_token;  /* [R] token in each row */
    int32_t* src_k;      /* [R] j of each row */
    int32_t* counts;     /* [P] copies per physical expert */
    int32_t* offsets;    /* [P+1] exclusive scan of counts */
    int32_t* error_word; /* [1] device error bits, shared by all sets */
    int32_t rows;        /* R */
    int32_t scale_stride;/* Gs */
} moe_view;

/*
 * The pool calls below serve the statically pre-allocated, double-buffered
 * per-expert buffers (write-up, "FusedDispatch and FusedCombine":
 * "Double-Buffered Static Pre-allocation"): buffers sized once for the worst
 * case, carved from one workspace, reused by every layer call.
 */

/*
 * Bytes of device workspace a pool with this geometry needs: every set's
 * dispatch and combine buffers at worst-case capacity ("Double-Buffered
 * Static Pre-allocation").  Host only.
 */
MOE_API int moe_pool_bytes(const moe_desc* desc, size_t* bytes);

/*
 * Create a pool over a caller-owned device workspace of at least
 * moe_pool_bytes(desc) bytes, 256-byte aligned.  The buffers are carved here
 * once and never allocated again ("Double-Buffered Static Pre-allocation").
 * Host only: nothing is launched and the workspace is not touched; call
 * moe_pool_clear_error once before first use.  The workspace must outlive
 * the pool.
 */
MOE_API int moe_pool_init(const moe_desc* desc, void* dev_ws, size_t ws_bytes, moe_pool** out);

/* Free the host handle; the workspace, and with it the pre-allocated buffers
 * ("Double-Buffered Static Pre-allocation"), stay the caller's. */
MOE_API int moe_pool_destroy(moe_pool* pool);

/* Device addresses of buffer set `buf`: its pre-allocated dispatch and
 * combine buffers and plan metadata ("Double-Buffered Static
 * Pre-allocation": one of the double-buffered sets). */
MOE_API int moe_pool_view(const moe_pool* pool, int buf, moe_view* view);

/*
 * Zero the device error word and the pool's plan tickets, the control block
 * in front of the pre-allocated sets ("Double-Buffered Static
 * Pre-allocation"), asynchronously on `stream`.  Call once before the pool's
 * first use, after any MOE_ERR_DEVICE, and never while the pool's kernels
 * run on another stream.
 */
MOE_API int moe_pool_clear_error(moe_pool* pool, void* stream);

/*
 * Synchronize `stream`, read the device error word into *error_word (may be
 * NULL) and return MOE_ERR_DEVICE if any bit is set, else MOE_OK.  The bits
 * record bad indices the kernels skipped instead of writing outside the
 * pre-allocated buffers ("Double-Buffered Static Pre-allocation").  The word
 * is not cleared.
 */
MOE_API int moe_pool_check(moe_pool* pool, void* stream, int32_t* error_word);

/* Number of kernels launched on this pre-allocated pool since init
 * ("Double-Buffered Static Pre-allocation"). */
MOE_API int moe_pool_launches(const moe_pool* pool, uint64_t* count);

/*
 * Host check of a replica map in CSR form: rep_off[0] = 0, every expert has
 * at least one replica, rep_off[E] = P, and rep_ids is a permutation of
 * [0, P) (each physical slot serves exactly one logical expert).  Host
 * pointers.  Returns MOE_OK or MOE_ERR_REPLICA.
 */
MOE_API int moe_replica_check(const int32_t* rep_off, const int32_t* rep_ids, int32_t E, int32_t P);

/*
 * moe_plan: routing metadata for T tokens into buffer set `buf`.
 *   logits   device fp32 [T, E] router logits
 *   rep_off  device int32 [E+1], rep_ids device int32 [P]: replica map (CSR);
 *            both NULL means physical = logical (requires P == E).
 * Per token t: the k largest logits (equal logits: lower expert id first),
 * gates = softmax over those k logits, the exact value rounded once to fp32
 * (except within about 2^-50 of an fp32 rounding midpoint), and the
 * physical replica rep_ids[rep_off[e] + t mod (rep_off[e+1] - rep_off[e])].
 * Then counts, offsets (exclusive scan, offsets[P] = T*k), slot[t,j] =
 * offsets[p] + (number of tokens before t routed to p), and the inverse
 * src_token / src_k.  Writes topk_e, gates, phys, counts, offsets, slot,
 * src_token, src_k of the set.  0 <= T <= T_max; T = 0 (an empty batch)
 * zeroes counts and offsets and launches no kernel (logits may be NULL).
 * Kernels: up to 512 tokens one thread-block cluster; beyond, three
 * launches (route, column scan, assign), routing tiles of 16 tokens up to
 * 2048 tokens when E > 128 or k > 16, else 32.  With the environment variable
 * MOE_PLAN_NO_CLUSTER=1 (read once per process), or on a device that refuses
 * the cluster, batches of up to 128 tokens take one launch whose last CTA
 * finishes the placement, and larger ones the three launches.  The results
 * do not depend on the form.
 */
MOE_API int moe_plan(moe_pool* pool, const float* logits, int32_t T,
                     const int32_t* rep_off, const int32_t* rep_ids, int buf, void* stream);

/*
 * moe_dispatch: quantize x and scatter into the set's dispatch rows
 * (write-up, "FusedDispatch and FusedCombine": "Early INT8 Quantization",
 * "AIV-Direct Write", "Token-Level Pipeline").
 *   x  device bf16 [T, H]
 * Per token and 128-element group g: amax = max |x|, scale = amax / 127 (fp32),
 * code = rint((x * 127) / amax) in fp32, half-even (amax = 0: scale 0, codes 0).
 * Row slot[t, j] of codes / scales receives token t's codes / scales for every
 * j.  Requires a prior moe_plan on this set with the same T (T = 0: no-op).
 * x may be written by anything earlier on `stream`, kernels included.
 */
MOE_API int moe_dispatch(moe_pool* pool, const uint16_t* x, int32_t T, int buf, void* stream);

/*
 * moe_dispatch_after_plan: moe_dispatch for the plan -> dispatch sequence,
 * with x loaded and quantized while the plan still runs (same passages, same
 * results, about half a microsecond earlier on a 96-token batch).  x is read
 * BEFORE the wait for the preceding kernel, so this is correct only when the
 * kernel enqueued just before this call on `stream` is this set's moe_plan
 * (which never writes x and lets its dependents start only after its own
 * wait), and x was written before that plan in stream order.  The library
 * cannot check this: with any other kernel in between (one that writes x, or
 * one launched with programmatic dependent launch that triggers its
 * dependents early), use moe_dispatch.  Arguments and errors as moe_dispatch.
 * moe_plan_dispatch gives the same early load with the precondition met by
 * construction.
 */
MOE_API int moe_dispatch_after_plan(moe_pool* pool, const uint16_t* x, int32_t T, int buf, void* stream);

/*
 * moe_plan_dispatch: moe_plan followed by moe_dispatch on set `buf` and
 * `stream`, as one call (write-up, "FusedDispatch and FusedCombine": the
 * routing metadata and the token data of one dispatch; "Token-Level
 * Pipeline").  Arguments and errors as the two calls; x is checked before
 * the plan is launched, so an error leaves nothing enqueued.  The results are
 * the same bit for bit.  Because the plan is then the kernel just before the
 * dispatch, the dispatch loads and quantizes x while the plan runs (as
 * moe_dispatch_after_plan does), and that is always safe here: x and the
 * logits may be written by anything earlier on `stream`, kernels included.
 * T = 0: as moe_plan (x may be NULL).
 */
MOE_API int moe_plan_dispatch(moe_pool* pool, const float* logits, int32_t T, const int32_t* rep_off,
                              const int32_t* rep_ids, const uint16_t* x, int buf, void* stream);

/*
 * Identity experts (test stand-in for the expert FFNs): for rows r < T*k,
 * ex_out[r, i] = bf16(codes[r, i] * scales[r, i/128]).  Requires a prior
 * moe_plan and moe_dispatch on this set with the same T.
 */
MOE_API int moe_identity_experts(moe_pool* pool, int32_t T, int buf, void* stream);

/*
 * moe_combine: y[t, i] = bf16( acc ), acc = 0, then for j = 0..k-1
 * acc = fmaf(gates[t, j], ex_out[slot[t, j], i], acc).
 *   ex_out  device bf16 [T*k (or more), H] expert outputs by row, or NULL to
 *           use the set's own ex_out buffer
 *   y       device bf16 [T, H] output
 * Requires a prior moe_plan on this set with the same T (T = 0: no-op).
 */
MOE_API int moe_combine(moe_pool* pool, const uint16_t* ex_out, uint16_t* y, int32_t T, int buf,
                        void* stream);

/*
 * One whole layer from HOST buffers: copy logits [T, E] and x [T, H] to the
 * device (into the set's staging area of the workspace), moe_plan_dispatch
 * (rep_off / rep_ids are DEVICE pointers, as for moe_plan), then either copy
 * h_ex_out [T*k, H] (bf16 expert outputs, by
 * row) into the set's ex_out buffer or, if h_ex_out is NULL, run
 * moe_identity_experts; then moe_combine and copy y [T, H] back to h_y.
 * All copies are cudaMemcpyAsync on `stream`; host buffers should be pinned.
 * The call returns once everything is enqueued: h_y is valid after the
 * stream is synchronized.  Uses the set's staging buffers, so calls on the
 * same set must not overlap.
 */
MOE_API int moe_step_host(moe_pool* pool, const float* h_logits, const uint16_t* h_x,
                          const uint16_t* h_ex_out, uint16_t* h_y, int32_t T,
                          const int32_t* rep_off, const int32_t* rep_ids, int buf, void* stream);

/*
 * moe_plan_static: moe_plan for callers that cannot allocate device memory.
 * The pages have no counterpart to this call; it exists because some callers
 * have no allocator to give the pool workspace: code replayed inside a CUDA
 * graph built elsewhere, plugins whose host framework owns every device
 * allocation, or processes that must not grow their device footprint after
 * start-up.
 *
 * Computes exactly what moe_plan computes (same kernels), into the caller's
 * own device arrays instead of a pool set:
 *   logits [T, E] fp32 in; topk_e, phys, slot int32 [T, k], gates fp32 [T, k],
 *   counts int32 [P], offsets int32 [P+1], src_token, src_k int32 [T*k] out;
 *   error_word int32 [1]: device error bits are OR-ed in (zero it first).
 *   rep_off / rep_ids: device replica map as for moe_plan, or both NULL (P == E).
 * Its scratch (per-tile expert counts and in-tile ranks) lives in a fixed
 * 4 MiB array in this library's device image, held on every GPU that loads it
 * until the process exits.  Sizes whose scratch needs more,
 * 4 * (P * ceil(T / TT) + T * k) bytes (each part rounded up to 256), return
 * MOE_ERR_SIZE before anything is launched; TT, the plan's tile, is 16 tokens
 * for batches of 513 to 2048 tokens with E > 128 or k > 16, else 32.  No
 * cudaMalloc or cudaFree is called.
 *   - All calls share that array: calls whose kernels overlap on the GPU
 *     (other streams, other host threads) race and give wrong slots.  Batches
 *     of up to 512 tokens take the cluster plan, which keeps its scratch in
 *     shared memory and does not touch the array, where the device launches
 *     clusters (not with MOE_PLAN_NO_CLUSTER=1).
 *     Where the device refuses the cluster launch, such a batch silently
 *     takes the three-launch plan, which does use the array.
 *   - The first call on each device (and again after the device's context is
 *     destroyed and re-created, e.g. by cudaDeviceReset) looks up the array's
 *     device address with that device current; make it before any stream
 *     capture begins.
 *   - Argument checks do not depend on T (except that logits may be NULL
 *     when T = 0): an empty batch passes the same checks and then only zeroes
 *     counts and offsets.
 */
MOE_API int moe_plan_static(const float* logits, int32_t T, int32_t E, int32_t P, int32_t k,
                            const int32_t* rep_off, const int32_t* rep_ids, int32_t* topk_e,
                            float* gates, int32_t* phys, int32_t* counts, int32_t* offsets,
                            int32_t* slot, int32_t* src_token, int32_t* src_k, int32_t* error_word,
                            void* stream);

/* Static string for a moe_status value, the status of the pool calls above
 * (write-up, "FusedDispatch and FusedCombine": "Double-Buffered Static
 * Pre-allocation"). */
MOE_API const char* moe_status_str(int status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
