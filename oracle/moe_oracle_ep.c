/*
 * moe_oracle_ep.c -- plain CPU oracle for the expert-parallel split of the
 * dispatch / combine pool over R ranks.
 *
 * TEST INFRASTRUCTURE ONLY, like moe_oracle.c: nothing on the product path
 * may link, load or call this file, and it shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes:
 *
 *   ownership  physical expert p lives on rank floor(p * R / P), so every rank
 *              owns one contiguous block of experts.
 *   layout     rank d's receive buffer is expert-major over its own experts;
 *              inside expert p's window come the rows of source rank 0, then
 *              rank 1, ..., each source's rows in the order of its own window
 *              (ascending token).  This is the StrataCL analysis, section 3.5:
 *              token placement -> expert-window aggregation -> peer-window
 *              partition, with the windows of one expert from every peer
 *              aggregated at its owner.
 *   gather     dispatch exchange: receiver d copies, for each of its experts
 *              and each source, the source's window rows into its own buffer
 *              (pull mode, StrataCL section 3.4: every rank reads the remote
 *              slices and writes its local buffer).
 *   return     combine exchange: source s copies its rows back from each
 *              owner's buffer into its own pool rows, where its local combine
 *              reads them (CloudMatrix384 write-up, "FusedDispatch and
 *              FusedCombine": expert output return).
 *   schedule   the transfer units of one puller and their assignment to C
 *              cores (StrataCL section 3.5): each (peer, expert) window is cut
 *              into units of at most S_t rows, unit cost tau = alpha_t +
 *              bytes / beta_t for the unit's tier t (0: the puller's own
 *              memory, 1: another rank's), and an LPT list scheduler --
 *              units by decreasing cost, each to the least-loaded core -- under
 *              the fan-out cap: in every stripe (the i-th unit of every core's
 *              list) at most H_t cores work on the same peer.
 *
 * Plain loops in that order; a library sort (qsort) orders the units.
 * Costs are integers (picoseconds): tau = alpha_ns * 1000 +
 * floor(bytes * 1000 / beta_gbs), so that ties are exact.
 * Every function returns 0 or a negative code (ORC_EP_ERR_ARG).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_EP_OK 0
#define ORC_EP_ERR_ARG (-1)

/* --------------------------------------------------------- ownership ---- */

int32_t orc_ep_owner(int32_t p, int32_t R, int32_t P) { return (int32_t)(((int64_t)p * R) / P); }

/* Number of experts rank d owns (found by scanning every expert). */
static int32_t orc_ep_count_owned(int32_t d, int32_t R, int32_t P) {
    int32_t n = 0;
    for (int32_t p = 0; p < P; ++p)
        if (orc_ep_owner(p, R, P) == d) n += 1;
    return n;
}

/* Start of expert p's window in source s's own pool: the sum of s's counts
 * of every expert before p (the exclusive scan of the plan). */
static int64_t orc_ep_pool_row(const int32_t* counts, int32_t P, int32_t s, int32_t p) {
    int64_t row = 0;
    for (int32_t q = 0; q < p; ++q) row += counts[(size_t)s * P + q];
    return row;
}

/* Start of source s's rows of expert p in its owner's receive buffer: every
 * row of the owner's earlier experts (all sources), then the rows of expert p
 * from sources before s. */
static int64_t orc_ep_recv_row(const int32_t* counts, int32_t R, int32_t P, int32_t s, int32_t p) {
    const int32_t d = orc_ep_owner(p, R, P);
    int64_t row = 0;
    for (int32_t q = 0; q < p; ++q) {
        if (orc_ep_owner(q, R, P) != d) continue;
        for (int32_t r = 0; r < R; ++r) row += counts[(size_t)r * P + q];
    }
    for (int32_t r = 0; r < s; ++r) row += counts[(size_t)r * P + p];
    return row;
}

/* ------------------------------------------------------------ layout ---- */

/*
 * Receive layout of rank d.
 *   counts      int32 [R, P]: counts[s, p] = rows source s routed to expert p
 *   n_experts   out: number of experts d owns (n_d)
 *   expert_off  int32 [n_d + 1]: start of each owned expert's window; the
 *               last entry is the number of rows d receives
 *   chunk_row   int32 [R, n_d]: start of source s's rows of the i-th owned
 *               expert
 * The arrays must hold P + 1 and R * P entries (any rank owns at most P).
 */
int orc_ep_layout(const int32_t* counts, int32_t R, int32_t P, int32_t d, int32_t* n_experts,
                  int32_t* expert_off, int32_t* chunk_row) {
    if (!counts || !n_experts || !expert_off || !chunk_row || R < 1 || P < 1 || d < 0 || d >= R)
        return ORC_EP_ERR_ARG;
    const int32_t nd = orc_ep_count_owned(d, R, P);
    int64_t row = 0;
    int32_t i = 0;
    for (int32_t p = 0; p < P; ++p) {
        if (orc_ep_owner(p, R, P) != d) continue;
        expert_off[i] = (int32_t)row;
        for (int32_t s = 0; s < R; ++s) {
            chunk_row[(size_t)s * nd + i] = (int32_t)row;
            row += counts[(size_t)s * P + p];
        }
        i += 1;
    }
    expert_off[nd] = (int32_t)row;
    *n_experts = nd;
    return ORC_EP_OK;
}

/* ------------------------------------------------------------ gather ---- */

/*
 * Dispatch exchange for receiver d, one plane (codes, scales, ...).
 *   src        R pointers: the plane of each source rank's pool (rows of
 *              row_bytes bytes, expert-major windows)
 *   dst        the plane of d's receive buffer
 * For each expert p that d owns, ascending, and each source s, ascending:
 * the counts[s, p] rows of s's window of p are appended to dst.
 */
int orc_ep_gather(const uint8_t* const* src, int64_t row_bytes, const int32_t* counts, int32_t R, int32_t P,
                  int32_t d, uint8_t* dst) {
    if (!src || !counts || !dst || row_bytes < 1 || R < 1 || P < 1 || d < 0 || d >= R) return ORC_EP_ERR_ARG;
    int64_t row = 0;
    for (int32_t p = 0; p < P; ++p) {
        if (orc_ep_owner(p, R, P) != d) continue;
        for (int32_t s = 0; s < R; ++s) {
            const int64_t n = counts[(size_t)s * P + p];
            const int64_t from = orc_ep_pool_row(counts, P, s, p);
            memcpy(dst + row * row_bytes, src[s] + from * row_bytes, (size_t)(n * row_bytes));
            row += n;
        }
    }
    return ORC_EP_OK;
}

/* ------------------------------------------------------------ return ---- */

/*
 * Combine exchange for source s, one plane: the inverse of the gather.
 *   recv       R pointers: the plane of each rank's receive buffer
 *   dst        the plane of s's own pool
 * For every expert p: the counts[s, p] rows at s's place in p's owner's
 * window go back to rows [pool_row(s, p), +counts[s, p]) of dst.
 */
int orc_ep_return(const uint8_t* const* recv, int64_t row_bytes, const int32_t* counts, int32_t R, int32_t P,
                  int32_t s, uint8_t* dst) {
    if (!recv || !counts || !dst || row_bytes < 1 || R < 1 || P < 1 || s < 0 || s >= R) return ORC_EP_ERR_ARG;
    for (int32_t p = 0; p < P; ++p) {
        const int32_t d = orc_ep_owner(p, R, P);
        const int64_t n = counts[(size_t)s * P + p];
        const int64_t from = orc_ep_recv_row(counts, R, P, s, p);
        const int64_t to = orc_ep_pool_row(counts, P, s, p);
        memcpy(dst + to * row_bytes, recv[d] + from * row_bytes, (size_t)(n * row_bytes));
    }
    return ORC_EP_OK;
}

/* ---------------------------------------------------------- schedule ---- */

typedef struct {
    int32_t peer, src_row, dst_row, rows;
} orc_ep_unit;

typedef struct {
    int64_t cost;
    int32_t index; /* position in the enumeration (ascending destination row) */
} orc_ep_key;

/* Larger cost first; equal costs in enumeration order. */
static int orc_ep_key_cmp(const void* pa, const void* pb) {
    const orc_ep_key* a = (const orc_ep_key*)pa;
    const orc_ep_key* b = (const orc_ep_key*)pb;
    if (a->cost > b->cost) return -1;
    if (a->cost < b->cost) return 1;
    return (a->index < b->index) ? -1 : (a->index > b->index);
}

/* Append the units of one window of n rows: pieces of at most S rows. */
static int orc_ep_split(orc_ep_unit* u, int32_t* nu, int32_t max_units, int32_t peer, int64_t src0, int64_t dst0,
                        int64_t n, int32_t S) {
    for (int64_t done = 0; done < n; done += S) {
        if (*nu >= max_units) return ORC_EP_ERR_ARG;
        const int64_t rows = (n - done < S) ? (n - done) : S;
        u[*nu].peer = peer;
        u[*nu].src_row = (int32_t)(src0 + done);
        u[*nu].dst_row = (int32_t)(dst0 + done);
        u[*nu].rows = (int32_t)rows;
        *nu += 1;
    }
    return ORC_EP_OK;
}

/*
 * The transfer schedule of one puller.
 *   direction  0: dispatch -- puller d pulls, from every source s, the rows of
 *              the experts d owns (src_row in s's pool, dst_row in d's
 *              receive buffer); 1: combine -- puller s pulls its rows back
 *              from every owner d (src_row in d's receive buffer, dst_row in
 *              s's pool).
 *   C          cores (worker CTAs) of the puller
 *   cap[t]     fan-out cap H_t; unit_rows[t] unit size S_t; alpha_ns[t],
 *              beta_gbs[t] the cost model, for tier t (0: peer == puller)
 *   row_bytes  bytes a row moves (all planes of the row together)
 * Units are enumerated in ascending destination row (windows cut into pieces
 * of S_t rows), costed, sorted by decreasing cost (ties: enumeration order),
 * and assigned one by one to the least-loaded eligible core (ties: lowest
 * core), where a core is eligible for a unit of peer q if fewer than
 * cap[tier(q)] cores already hold a unit of q at that core's next stripe.
 * Outputs: units [n_units] grouped by core (core c's list, in the order it
 * was assigned, is units[core_off[c] .. core_off[c+1])), cost [n_units] in
 * the same order (ps), core_off [C+1], and the makespan (largest core load).
 */
int orc_ep_schedule(int32_t direction, int32_t puller, const int32_t* counts, int32_t R, int32_t P, int32_t C,
                    const int32_t* cap, const int32_t* unit_rows, const int64_t* alpha_ns, const int64_t* beta_gbs,
                    int64_t row_bytes, int32_t max_units, orc_ep_unit* units, int64_t* cost, int32_t* n_units,
                    int32_t* core_off, int64_t* makespan) {
    if (!counts || !cap || !unit_rows || !alpha_ns || !beta_gbs || !units || !cost || !n_units || !core_off ||
        !makespan || (direction != 0 && direction != 1) || R < 1 || P < 1 || puller < 0 || puller >= R || C < 1 ||
        row_bytes < 1 || max_units < 0)
        return ORC_EP_ERR_ARG;
    for (int t = 0; t < 2; ++t)
        if (cap[t] < 1 || unit_rows[t] < 1 || alpha_ns[t] < 0 || beta_gbs[t] < 1) return ORC_EP_ERR_ARG;

    /* 1. enumerate the units in ascending destination row */
    orc_ep_unit* u = (orc_ep_unit*)malloc(sizeof(orc_ep_unit) * (size_t)(max_units > 0 ? max_units : 1));
    if (!u) return ORC_EP_ERR_ARG;
    int32_t nu = 0;
    int rc = ORC_EP_OK;
    if (direction == 0) {
        const int32_t d = puller;
        for (int32_t p = 0; p < P && rc == ORC_EP_OK; ++p) {
            if (orc_ep_owner(p, R, P) != d) continue;
            for (int32_t s = 0; s < R && rc == ORC_EP_OK; ++s)
                rc = orc_ep_split(u, &nu, max_units, s, orc_ep_pool_row(counts, P, s, p),
                                  orc_ep_recv_row(counts, R, P, s, p), counts[(size_t)s * P + p],
                                  unit_rows[s == d ? 0 : 1]);
        }
    } else {
        const int32_t s = puller;
        for (int32_t p = 0; p < P && rc == ORC_EP_OK; ++p) {
            const int32_t d = orc_ep_owner(p, R, P);
            rc = orc_ep_split(u, &nu, max_units, d, orc_ep_recv_row(counts, R, P, s, p),
                              orc_ep_pool_row(counts, P, s, p), counts[(size_t)s * P + p],
                              unit_rows[d == s ? 0 : 1]);
        }
    }
    if (rc != ORC_EP_OK) {
        free(u);
        return rc;
    }

    /* 2. cost of every unit: alpha + bytes / beta, in picoseconds */
    orc_ep_key* key = (orc_ep_key*)malloc(sizeof(orc_ep_key) * (size_t)(nu > 0 ? nu : 1));
    int64_t* load = (int64_t*)calloc((size_t)C, sizeof(int64_t));
    int32_t* len = (int32_t*)calloc((size_t)C, sizeof(int32_t));
    int32_t* owner_core = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nu > 0 ? nu : 1));
    int32_t* pos = (int32_t*)malloc(sizeof(int32_t) * (size_t)(nu > 0 ? nu : 1));
    /* stripe_peer[i * R + q]: cores whose i-th unit is from peer q */
    int32_t* stripe_peer = (int32_t*)calloc((size_t)(nu > 0 ? nu : 1) * (size_t)R, sizeof(int32_t));
    if (!key || !load || !len || !owner_core || !pos || !stripe_peer) {
        free(u); free(key); free(load); free(len); free(owner_core); free(pos); free(stripe_peer);
        return ORC_EP_ERR_ARG;
    }
    for (int32_t i = 0; i < nu; ++i) {
        const int t = (u[i].peer == puller) ? 0 : 1;
        const int64_t bytes = (int64_t)u[i].rows * row_bytes;
        key[i].cost = alpha_ns[t] * 1000 + (bytes * 1000) / beta_gbs[t];
        key[i].index = i;
    }

    /* 3. longest first */
    qsort(key, (size_t)nu, sizeof(orc_ep_key), orc_ep_key_cmp);

    /* 4. list scheduling under the fan-out cap */
    for (int32_t k = 0; k < nu; ++k) {
        const int32_t i = key[k].index;
        const int32_t q = u[i].peer;
        const int t = (q == puller) ? 0 : 1;
        int32_t best = -1;
        for (int32_t c = 0; c < C; ++c) {
            if (stripe_peer[(size_t)len[c] * R + q] >= cap[t]) continue;
            if (best < 0 || load[c] < load[best]) best = c;
        }
        /* a core with the longest list is always eligible (its next stripe is
           still empty), so best >= 0 */
        owner_core[i] = best;
        pos[i] = len[best];
        stripe_peer[(size_t)len[best] * R + q] += 1;
        len[best] += 1;
        load[best] += key[k].cost;
    }

    /* 5. group by core, each core's units in the order they were assigned */
    core_off[0] = 0;
    for (int32_t c = 0; c < C; ++c) core_off[c + 1] = core_off[c] + len[c];
    int64_t* cost_of = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nu > 0 ? nu : 1));
    if (!cost_of) {
        free(u); free(key); free(load); free(len); free(owner_core); free(pos); free(stripe_peer);
        return ORC_EP_ERR_ARG;
    }
    for (int32_t k = 0; k < nu; ++k) cost_of[key[k].index] = key[k].cost;
    for (int32_t i = 0; i < nu; ++i) {
        const int32_t at = core_off[owner_core[i]] + pos[i];
        units[at] = u[i];
        cost[at] = cost_of[i];
    }
    int64_t ms = 0;
    for (int32_t c = 0; c < C; ++c)
        if (load[c] > ms) ms = load[c];
    *makespan = ms;
    *n_units = nu;
    free(u); free(key); free(load); free(len); free(owner_core); free(pos); free(stripe_peer); free(cost_of);
    return ORC_EP_OK;
}
