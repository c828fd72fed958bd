/*
 * moe_ep.h -- C ABI of libmoe, part 2: the expert-parallel split of the
 * dispatch / combine pool over R ranks.
 *
 * The method's real setting (CloudMatrix384 write-up, "FusedDispatch and
 * FusedCombine"; StrataCL analysis, sections 3.4 and 3.5) spreads the
 * experts over the ranks of an expert-parallel group.  Here:
 *   - physical expert p lives on rank floor(p * R / P), one contiguous block
 *     of experts per rank (moe_ep_experts);
 *   - every rank plans and dispatches its own batch into its own pool with
 *     moe_plan / moe_dispatch (include/moe.h): its pool is expert-major, so
 *     the rows for rank d's experts form one contiguous peer window;
 *   - rank d's receive buffer is expert-major over d's experts: inside expert
 *     p's window come source rank 0's rows, then rank 1's, ..., each source's
 *     rows in its own window order (token placement -> expert-window
 *     aggregation -> peer-window partition, StrataCL section 3.5)
 *     (moe_ep_layout);
 *   - each direction is one pull exchange (StrataCL section 3.4: every rank
 *     reads remote slices into its own buffer; no producer-consumer
 *     handshake): receivers pull their experts' INT8 rows and scales from
 *     the sources (dispatch), then sources pull their bf16 expert outputs
 *     back into their own pool rows (combine), where moe_combine reduces
 *     them in ascending j as on one GPU;
 *   - a pull is cut into transfer units of at most S_t rows (one expert
 *     window of one peer per unit or less), each costed tau = alpha_t +
 *     bytes / beta_t for its tier t (0: the puller's own memory, 1: another
 *     rank's), and list-scheduled longest first onto C cores (worker CTAs),
 *     each unit to the least-loaded core, under the per-peer fan-out cap: in
 *     every stripe (the i-th unit of every core's list) at most H_t cores
 *     work on one peer (StrataCL section 3.5, min-makespan with a fairness
 *     constraint, LPT list scheduler) (moe_ep_schedule);
 *   - moe_ep_pull executes the units: for one puller on a real group (its
 *     peers' buffers mapped into its address space), or for all R pullers
 *     of a group emulated on one GPU in one launch, with every rank's
 *     buffers in local memory;
 *   - or, fused (the write-up's direct writes into the receivers'
 *     pre-allocated buffers): every (source, expert) window's first row in
 *     its owner's buffer comes from every rank's counts (moe_ep_recv_start on
 *     the host, moe_ep_recv_start_device without a trip to it);
 *     moe_ep_dispatch quantizes a rank's tokens once and writes each copy
 *     straight to its row in the owner's receive buffer, recording where it
 *     went; moe_ep_combine reads each copy's expert output where its owner
 *     holds it and reduces in ascending j into the rank's y (the reduction
 *     form of StrataCL section 3.4).  No schedule and no pull; the receive
 *     buffers and y are those of the pulled form, bit for bit.
 *
 * Conventions as in moe.h: 0 or a negative moe_status; arguments checked on
 * the host before anything is launched; device pointers 16-byte aligned;
 * every launch asynchronous on `stream`.  The host calls (experts, layout,
 * max_units, schedule) need no GPU and allocate only host memory.
 */
#ifndef MOE_EP_H
#define MOE_EP_H

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_EP_MAX_RANKS 64

/* Device error-word bit (moe_ep_pull, moe_ep_dispatch, moe_ep_combine): a
 * unit or a row outside its buffers, or an out-of-range peer, was skipped. */
#define MOE_DEVERR_UNIT 0x8

/*
 * The expert-parallel group and its transfer cost model (StrataCL section
 * 3.5).  Index t of the two-element arrays is the tier: 0 for units the
 * puller reads from its own memory, 1 for units read from another rank.
 *   R            ranks, 1 .. MOE_EP_MAX_RANKS
 *   P            physical experts, 1 .. 4096 (a rank may own none when P < R)
 *   cores        C, worker CTAs of one puller, 1 .. 4096
 *   fanout_cap   H_t >= 1: cores of one puller working on one peer in one stripe
 *   unit_rows    S_t: rows per transfer unit at most, 1 .. 2^20
 *   alpha_ns     per-unit latency of tier t in ns, 0 .. 2^40
 *   beta_gbs     bandwidth of tier t in GB/s (bytes per ns), >= 1
 * Unit cost in picoseconds: alpha_ns * 1000 + floor(bytes * 1000 / beta_gbs).
 */
typedef struct moe_ep_desc {
    int32_t R, P, cores;
    int32_t fanout_cap[2];
    int32_t unit_rows[2];
    int64_t alpha_ns[2];
    int64_t beta_gbs[2];
} moe_ep_desc;

/* One transfer unit (the remote-slice tuple <peer, src, dst, bytes> of
 * StrataCL section 3.4, in rows): rows [src_row, src_row + rows) of the
 * peer's source buffer go to rows [dst_row, dst_row + rows) of the puller's
 * destination buffer.  16 bytes. */
typedef struct moe_ep_unit {
    int32_t peer, src_row, dst_row, rows;
} moe_ep_unit;

/*
 * Experts of rank d: p in [*first, *first + *count), i.e. every p with
 * floor(p * R / P) == d (StrataCL section 3.5, expert windows aggregated at
 * their owner).  Host only.
 */
MOE_API int moe_ep_experts(int32_t R, int32_t P, int32_t d, int32_t* first, int32_t* count);

/*
 * Receive layout of rank d (StrataCL section 3.5: expert-window aggregation,
 * peer-window partition).
 *   counts      host int32 [R, P]: counts[s, p] = rows rank s routed to
 *               physical expert p (each rank's moe_plan counts)
 *   expert_off  host int32 [n_d + 1]: start row of each of d's experts in
 *               d's receive buffer; expert_off[n_d] = rows d receives
 *   chunk_row   host int32 [R, n_d]: start row of source s's rows of d's
 *               i-th expert (n_d = count from moe_ep_experts)
 * Host only.
 */
MOE_API int moe_ep_layout(int32_t R, int32_t P, const int32_t* counts, int32_t d, int32_t* expert_off,
                          int32_t* chunk_row);

/*
 * An upper bound on the units one puller's schedule can hold when it moves
 * at most `rows` rows: rows / min(S_t) + R * (experts of the largest rank).
 * Host only.
 */
MOE_API int moe_ep_max_units(const moe_ep_desc* desc, int64_t rows, int32_t* max_units);

/*
 * The transfer schedule of one puller (StrataCL section 3.5).
 *   direction  0 = dispatch: puller d pulls, from every rank s, s's rows of
 *              d's experts (src_row in s's pool rows, dst_row in d's receive
 *              buffer); 1 = combine: puller s pulls its rows back from every
 *              owner d (src_row in d's receive buffer, dst_row in s's pool
 *              rows)
 *   counts     host int32 [R, P] as for moe_ep_layout
 *   row_bytes  bytes one row moves (all planes together), 1 .. 2^24
 * Units are enumerated in ascending destination row (each (peer, expert)
 * window cut into pieces of at most S_t rows), costed, ordered by
 * decreasing cost (equal costs in enumeration order), and assigned one by
 * one to the least-loaded core among those whose next stripe holds fewer
 * than H_t units of the unit's peer (equal loads: the lower core; a core
 * with the longest list is always eligible).
 * Outputs (host): units [*n_units] grouped by core -- core c's list, in the
 * order assigned, is units[core_off[c] .. core_off[c+1]) -- core_off
 * [cores + 1], and the makespan (the largest core load, ps; may be NULL).
 * MOE_ERR_SIZE if more than max_units units are needed.  Host only.
 */
MOE_API int moe_ep_schedule(const moe_ep_desc* desc, int32_t direction, int32_t puller, const int32_t* counts,
                            int64_t row_bytes, moe_ep_unit* units, int32_t max_units, int32_t* n_units,
                            int32_t* core_off, int64_t* makespan_ps);

/*
 * The schedules of all R pullers of a group in one call (the same schedule
 * moe_ep_schedule gives each puller), computed on host worker threads the
 * library starts on first use and keeps until the process exits (a call made
 * while another one uses them, or in a process forked after they started,
 * computes on the calling thread), and packed: puller r's core c runs units[core_off[r, c] .. core_off[r, c+1])
 * with absolute indices, ready for moe_ep_pull with first_puller 0 and
 * n_pullers R.
 *   units        host moe_ep_unit [max_units] (all pullers together)
 *   core_off     host int32 [R, cores + 1]
 *   n_units      total units written
 *   makespan_ps  host int64 [R] (may be NULL)
 * MOE_ERR_SIZE if more than max_units units are needed in total (R times
 * moe_ep_max_units for the group's total rows always suffices).  Host only.
 */
MOE_API int moe_ep_schedule_group(const moe_ep_desc* desc, int32_t direction, const int32_t* counts,
                                  int64_t row_bytes, moe_ep_unit* units, int32_t max_units, int32_t* n_units,
                                  int32_t* core_off, int64_t* makespan_ps);

/*
 * One plane of a pull (INT8 codes, fp32 scales or bf16 rows): where the
 * plane lives in every rank's source and destination buffer.
 *   src[q], src_rows[q]  device address and row count of peer q's source
 *                        buffer (q < R)
 *   dst[r], dst_rows[r]  device address and row count of puller r's
 *                        destination buffer (r < R)
 *   row_bytes            bytes per row, a multiple of 16
 * Entries of ranks that take no part may be NULL with 0 rows.
 */
typedef struct moe_ep_plane {
    const void* src[MOE_EP_MAX_RANKS];
    void* dst[MOE_EP_MAX_RANKS];
    int64_t src_rows[MOE_EP_MAX_RANKS];
    int64_t dst_rows[MOE_EP_MAX_RANKS];
    int64_t row_bytes;
} moe_ep_plane;

/*
 * Execute the schedules of pullers first_puller .. first_puller + n_pullers - 1
 * in one launch (pull mode, StrataCL section 3.4): CTA (c, i) runs core c of
 * puller first_puller + i, its units in list order, copying every plane of
 * each unit (a contiguous run of rows in both buffers).
 *   units     device moe_ep_unit array holding every puller's list
 *   core_off  device int32 [n_pullers, cores + 1]: puller i's core c runs
 *             units[core_off[i, c] .. core_off[i, c + 1]) (absolute indices)
 *   n_units   entries in `units` (bound for the core_off entries)
 *   planes    host array of n_planes (1 or 2) plane descriptions
 *   error_word device int32: MOE_DEVERR_UNIT is OR-ed in for every unit that
 *             would reach outside a buffer or names a peer >= R; such a unit
 *             is skipped (no access made)
 * The launch waits (griddepcontrol.wait) for the kernel before it on
 * `stream` before reading anything.  Every source row must have been written
 * before: on one GPU, earlier in stream order; across GPUs, the caller
 * orders the peers' writes before this call.  n_pullers = 1 is a rank of a
 * real group; n_pullers = R pulls for a whole group emulated on one GPU
 * (every pointer local).
 */
MOE_API int moe_ep_pull(const moe_ep_unit* units, const int32_t* core_off, int32_t n_units, int32_t R,
                        int32_t cores, int32_t first_puller, int32_t n_pullers, const moe_ep_plane* planes,
                        int32_t n_planes, int32_t* error_word, void* stream);

/*
 * Where rank s's copies of each expert sit in the expert's owner's receive
 * buffer (StrataCL section 3.5 layout, as moe_ep_layout):
 *   recv_start  host int32 [P]: for physical expert p owned by rank d, the
 *               first row of source s's window of p in d's receive buffer
 * (0 where s routed nothing to p).  Host only.
 */
MOE_API int moe_ep_recv_start(int32_t R, int32_t P, const int32_t* counts, int32_t s, int32_t* recv_start);

/*
 * moe_ep_recv_start on the device, for every rank at once, from the ranks'
 * counts where the plans left them (no trip to the host):
 *   counts      host array [R] of device addresses: rank q's int32 [P] counts
 *   recv_start  device int32 [R, P]: row s is rank s's moe_ep_recv_start
 *   recv_rows   device int32 [R]: rows each rank receives (may be NULL)
 * (int32 tables of this header need 4-byte alignment only.)
 * One launch of one CTA; it waits for the kernel before it (the plans) before
 * reading the counts.
 */
MOE_API int moe_ep_recv_start_device(int32_t R, int32_t P, const int32_t* const* counts, int32_t* recv_start,
                                     int32_t* recv_rows, void* stream);

/*
 * Fused dispatch of rank s (CloudMatrix384 write-up, "FusedDispatch and
 * FusedCombine": each token quantized once and its rows written directly into
 * the receivers' pre-allocated buffers, "AIV-Direct Write", in a token-level
 * load -> quantize/address -> write pipeline).  Quantizes x as moe_dispatch
 * does and writes copy (t, j) -- expert p = phys[t, j], owner floor(p R / P)
 * -- to row recv_start[p] + slot[t, j] - offsets[p] of the owner's receive
 * buffer, codes and scales, instead of the pool's own rows.  The receive
 * buffers then hold exactly what moe_ep_pull (direction 0) would gather.
 *   x            device bf16 [T, H] (read after the wait for the kernel before)
 *   recv_codes   host array [R] of device addresses: each owner's int8 [rows, H]
 *   recv_scales  host array [R] of device addresses: each owner's fp32
 *                [rows, Gs] (Gs = the pool's scale stride, moe_view)
 *   recv_rows    host int64 [R]: rows each owner's buffers hold (bounds)
 *   recv_start   device int32 [P]: this rank's row of moe_ep_recv_start(_device),
 *                4-byte aligned
 *   copy_row     device int64 [T, k] or NULL: where each copy went, recorded
 *                for moe_ep_combine -- owner * 2^40 + row, or -1 for a copy
 *                that was skipped; 8-byte aligned
 * A row outside its owner's buffer is skipped and sets MOE_DEVERR_UNIT.
 * Requires a prior moe_plan on this set with the same T.
 */
MOE_API int moe_ep_dispatch(moe_pool* pool, const uint16_t* x, int32_t T, int buf, int32_t R,
                            int8_t* const* recv_codes, float* const* recv_scales, const int64_t* recv_rows,
                            const int32_t* recv_start, int64_t* copy_row, void* stream);

/*
 * Fused combine of rank s (a pull-mode reduction, StrataCL section 3.4:
 * remote operands loaded on chip and accumulated into the local output;
 * CloudMatrix384 write-up, "FusedDispatch and FusedCombine": expert output
 * return and weighted reduce in one operator).  For every token t of the
 * pool's set `buf` (planned with T tokens on rank s), and j = 0..k-1 in
 * ascending order, the copy's expert output row is read straight from its
 * owner's receive buffer -- row recv_start[p] + slot[t, j] - offsets[p] of
 * rank floor(p * R / P)'s buffer, p = phys[t, j] -- and accumulated with
 * fmaf(gate, row, acc) in fp32; y[t] = bf16(acc).  The result equals a
 * combine pull (moe_ep_pull, direction 1) followed by moe_combine, bit for
 * bit, without writing the rows back.
 *   recv_ex    host array [R] of device addresses: each owner's bf16 [rows, H]
 *              expert outputs (NULL with 0 rows for a rank that owns none)
 *   recv_rows  host int64 [R]: rows of each owner's buffer (bounds)
 *   recv_start device int32 [P] (moe_ep_recv_start of rank s), 4-byte aligned
 *   copy_row   device int64 [T, k] or NULL: the rows moe_ep_dispatch recorded
 *              for this set and batch (then recv_start is not read and may be
 *              NULL); with NULL each row is found from phys, offsets and
 *              recv_start, one dependent load more per copy
 *   y          device bf16 [T, H]
 * A row outside its owner's buffer (or a recorded -1) skips the token's
 * segment and sets MOE_DEVERR_UNIT in the pool's error word.  Requires a
 * prior moe_plan on this set with the same T.
 */
MOE_API int moe_ep_combine(moe_pool* pool, int32_t T, int buf, int32_t R, const uint16_t* const* recv_ex,
                           const int64_t* recv_rows, const int32_t* recv_start, const int64_t* copy_row,
                           uint16_t* y, void* stream);

/*
 * Dequantize rows (the identity-expert stand-in on any buffer, e.g. a
 * receive buffer): out[r, i] = bf16(codes[r, i] * scales[r, i / 128]) for
 * r < rows (CloudMatrix384 write-up, "FusedDispatch and FusedCombine": INT8
 * codes with their scale factor).
 *   codes  device int8 [rows, H]; scales device fp32 [rows, scale_stride]
 *   out    device bf16 [rows, H]; H a multiple of 128, scale_stride >= H/128
 *          and a multiple of 4
 */
MOE_API int moe_dequant_rows(const int8_t* codes, const float* scales, int32_t rows, int32_t H,
                             int32_t scale_stride, uint16_t* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_EP_H */
