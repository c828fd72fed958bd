/*
 * moe_oracle.c -- plain CPU oracle for MoE FusedDispatch / FusedCombine.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it exists so that tests, the smoke check and the bench's
 * CPU baseline can compare the CUDA library against an independent,
 * obviously-correct implementation.  It shares no code, header, table or
 * helper with the CUDA library.
 *
 * What it computes (CloudMatrix384 write-up, section "FusedDispatch and
 * FusedCombine"; "Decode Phase"; "Prefill Phase" for metadata generation;
 * StrataCL analysis section 3.5 for the token-placement -> expert-window
 * hierarchy):
 *
 *   route     per token: the k largest router logits (ties -> lower expert id),
 *             gates = softmax over those k logits, each logical expert mapped to
 *             a physical slot through the redundant-replica map.
 *   plan      histogram of physical experts, exclusive scan into expert
 *             windows, stable (ascending token) placement of every (token, j)
 *             copy inside its expert's window, and the inverse map.
 *   dispatch  per token and per 128-element group: amax, fp32 scale
 *             amax/127, INT8 codes rint(x*127/amax); the codes and scales are
 *             written into each of the token's k slots.
 *   experts   identity experts for the round-trip check: bf16(code * scale).
 *   combine   per token: y = bf16( fma-chain over j ascending of
 *             gate_j * expert_row_j ), accumulated in fp32.
 *
 * Precision follows the fixed numerics of the method where they are stated
 * (fp32 quantization, fp32 fma accumulation, bf16 rounding).  Where the pages
 * leave it open -- the gate softmax -- the oracle computes in fp64 and rounds
 * once to fp32.
 *
 * Plain loops, one step after another, no blocking or fusion.  Every function
 * returns 0 on success or a negative code for inputs outside the method's
 * domain (outputs are then unspecified).  Build: gcc -std=c11 -O2
 * -ffp-contract=off -fPIC -shared -lm, plus -fopenmp where the compiler has
 * it: the per-token loops (route, quantize, dispatch, experts, combine) then
 * split their tokens over threads.  Each token's arithmetic is the same in
 * either build, so the results are identical; the counting sort stays serial.
 * When several tokens are bad, the lowest token's error code is returned, as
 * a serial loop would.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_REPLICA (-2)
#define ORC_ERR_DUPLICATE (-3)
#define ORC_ERR_NONFINITE (-4)

/* ------------------------------------------------------------ threads ---- */

/* Threads the per-token loops use (1 without OpenMP).  n < 1 leaves it as is. */
int orc_set_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* Record a failing token; the lowest token index keeps its code. */
static void orc_note_error(int32_t t, int rc, int32_t* err_t, int* err_rc) {
#pragma omp critical(orc_error)
    {
        if (*err_t < 0 || t < *err_t) {
            *err_t = t;
            *err_rc = rc;
        }
    }
}

/* ---------------------------------------------------------------- bf16 ---- */

/* bf16 is the upper half of an IEEE binary32: widening is exact. */
static float orc_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bf16, round to nearest, ties to even; NaN stays NaN (quiet). */
static uint16_t orc_f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t keep = u >> 16;
    uint32_t rest = u & 0xffffu;
    if (rest > 0x8000u || (rest == 0x8000u && (keep & 1u))) keep += 1u;
    return (uint16_t)keep;
}

/* ----------------------------------------------------------- route (a1-a3) */

typedef struct {
    float v;
    int32_t e;
} orc_cand;

/* Order: larger logit first; equal logits -> smaller expert id first. */
static int orc_cand_cmp(const void* pa, const void* pb) {
    const orc_cand* a = (const orc_cand*)pa;
    const orc_cand* b = (const orc_cand*)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->e < b->e) ? -1 : (a->e > b->e);
}

/*
 * Top-k routing, gate softmax and replica pick for T tokens.
 *   logits   fp32 [T, E] row-major
 *   rep_off  int32 [E+1] CSR offsets into rep_ids, or NULL for phys = expert
 *   rep_ids  int32 [P]   physical ids of each expert's replicas
 * Outputs, all [T, k] row-major: topk_e (logical expert), gates (fp32), phys.
 *
 * Gates: m = the top logit; e_j = exp(l_j - m) and s = e_0 + ... + e_{k-1}
 * in fp64, ascending j; gate_j = (float)(e_j / s).
 * Replica: the token at index t picks replica t mod (replica count).
 */
static int orc_route_token(const float* row, int32_t t, int32_t E, int32_t k,
                           const int32_t* rep_off, const int32_t* rep_ids, int32_t P,
                           orc_cand* c, double* ex,
                           int32_t* topk_e, float* gates, int32_t* phys) {
    for (int32_t e = 0; e < E; ++e) {
        if (!isfinite(row[e])) return ORC_ERR_NONFINITE;
        c[e].v = row[e];
        c[e].e = e;
    }
    qsort(c, (size_t)E, sizeof(orc_cand), orc_cand_cmp);

    double s = 0.0;
    for (int32_t j = 0; j < k; ++j) {
        ex[j] = exp((double)c[j].v - (double)c[0].v);
        s += ex[j];
    }
    for (int32_t j = 0; j < k; ++j) {
        int32_t e = c[j].e;
        int32_t p = e;
        if (rep_off) {
            int32_t lo = rep_off[e], n = rep_off[e + 1] - rep_off[e];
            if (n < 1 || lo < 0 || lo + n > P) return ORC_ERR_REPLICA;
            p = rep_ids[lo + (t % n)];
            if (p < 0 || p >= P) return ORC_ERR_REPLICA;
        }
        topk_e[j] = e;
        gates[j] = (float)(ex[j] / s);
        phys[j] = p;
    }
    return ORC_OK;
}

int orc_route(const float* logits, int32_t T, int32_t E, int32_t k,
              const int32_t* rep_off, const int32_t* rep_ids, int32_t P,
              int32_t* topk_e, float* gates, int32_t* phys) {
    if (!logits || !topk_e || !gates || !phys || T < 0 || E < 1 || k < 1 || k > E || P < E)
        return ORC_ERR_ARG;
    int32_t err_t = -1;
    int err_rc = ORC_OK;
#pragma omp parallel
    {
        orc_cand* c = (orc_cand*)malloc(sizeof(orc_cand) * (size_t)E);
        double* ex = (double*)malloc(sizeof(double) * (size_t)k);
#pragma omp for schedule(static)
        for (int32_t t = 0; t < T; ++t) {
            int rc = (c && ex) ? orc_route_token(logits + (size_t)t * E, t, E, k, rep_off, rep_ids, P, c, ex,
                                                 topk_e + (size_t)t * k, gates + (size_t)t * k,
                                                 phys + (size_t)t * k)
                               : ORC_ERR_ARG;
            if (rc != ORC_OK) orc_note_error(t, rc, &err_t, &err_rc);
        }
        free(c);
        free(ex);
    }
    return err_rc;
}

/* ------------------------------------------------------ placement (a4-a6) */

/*
 * Counting sort of the T*k (token, j) copies by physical expert.
 *   counts[p]   copies routed to physical expert p              int32 [P]
 *   offsets[p]  start of expert p's window; offsets[P] = T*k       int32 [P+1]
 *   slot[t,j]   row of copy (t, j): offsets[p] + number of tokens before t
 *               routed to p (ascending token order)               int32 [T, k]
 *   src_token[r], src_k[r]  inverse: which (t, j) sits in row r    int32 [T*k]
 * A token routed twice to one physical expert is outside the method (a
 * well-formed replica map cannot produce it) and returns ORC_ERR_DUPLICATE.
 */
int orc_place(const int32_t* phys, int32_t T, int32_t k, int32_t P,
              int32_t* counts, int32_t* offsets, int32_t* slot,
              int32_t* src_token, int32_t* src_k) {
    if (!phys || !counts || !offsets || !slot || !src_token || !src_k || T < 0 || k < 1 || P < 1)
        return ORC_ERR_ARG;
    for (int32_t p = 0; p < P; ++p) counts[p] = 0;
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < k; ++j) {
            int32_t p = phys[(size_t)t * k + j];
            if (p < 0 || p >= P) return ORC_ERR_ARG;
            for (int32_t i = 0; i < j; ++i)
                if (phys[(size_t)t * k + i] == p) return ORC_ERR_DUPLICATE;
            counts[p] += 1;
        }
    }
    offsets[0] = 0;
    for (int32_t p = 0; p < P; ++p) offsets[p + 1] = offsets[p] + counts[p];

    int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)P);
    if (!cursor) return ORC_ERR_ARG;
    for (int32_t p = 0; p < P; ++p) cursor[p] = offsets[p];
    for (int32_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < k; ++j) {
            int32_t p = phys[(size_t)t * k + j];
            int32_t r = cursor[p];
            cursor[p] += 1;
            slot[(size_t)t * k + j] = r;
            src_token[r] = t;
            src_k[r] = j;
        }
    }
    free(cursor);
    return ORC_OK;
}

/* ------------------------------------------------------- dispatch (a7-a8) */

/*
 * Per-token INT8 quantization with one fp32 scale per 128-element group.
 *   x       bf16 bits [T, H]
 *   codes   int8 [T, H]
 *   scales  fp32 [T, H/128]
 * amax = max |x| over the group; scale = amax / 127 (fp32);
 * code = rint((x * 127) / amax) in fp32, round-half-even; amax == 0 gives
 * scale 0 and all-zero codes.  |x| <= amax makes |code| <= 127.
 */
static int orc_quantize_token(const uint16_t* x, int32_t H, int8_t* codes, float* scales) {
    const int32_t G = H / 128;
    for (int32_t g = 0; g < G; ++g) {
        const uint16_t* xs = x + (size_t)g * 128;
        float amax = 0.0f;
        for (int32_t i = 0; i < 128; ++i) {
            float v = orc_bf16_to_f32(xs[i]);
            if (!isfinite(v)) return ORC_ERR_NONFINITE;
            float a = fabsf(v);
            if (a > amax) amax = a;
        }
        scales[g] = amax / 127.0f;
        for (int32_t i = 0; i < 128; ++i) {
            int8_t q = 0;
            if (amax > 0.0f) {
                float v = orc_bf16_to_f32(xs[i]);
                float num = v * 127.0f;
                float quo = num / amax;
                q = (int8_t)(int32_t)rintf(quo);
            }
            codes[(size_t)g * 128 + i] = q;
        }
    }
    return ORC_OK;
}

int orc_quantize(const uint16_t* x, int32_t T, int32_t H,
                 int8_t* codes, float* scales) {
    if (!x || !codes || !scales || T < 0 || H < 128 || H % 128 != 0) return ORC_ERR_ARG;
    const int32_t G = H / 128;
    int32_t err_t = -1;
    int err_rc = ORC_OK;
#pragma omp parallel for schedule(static)
    for (int32_t t = 0; t < T; ++t) {
        int rc = orc_quantize_token(x + (size_t)t * H, H, codes + (size_t)t * H, scales + (size_t)t * G);
        if (rc != ORC_OK) orc_note_error(t, rc, &err_t, &err_rc);
    }
    return err_rc;
}

/*
 * Dispatch = quantize each token once, then write its codes and scales into
 * every one of its k slots.
 *   slot          int32 [T, k] from orc_place
 *   pool_codes    int8 [R, H]      rows R >= T*k
 *   pool_scales   fp32 [R, H/128]
 */
int orc_dispatch(const uint16_t* x, int32_t T, int32_t H, int32_t k,
                 const int32_t* slot, int32_t R,
                 int8_t* pool_codes, float* pool_scales) {
    if (!x || !slot || !pool_codes || !pool_scales || T < 0 || k < 1 || H < 128 || H % 128 != 0)
        return ORC_ERR_ARG;
    const int32_t G = H / 128;
    int32_t err_t = -1;
    int err_rc = ORC_OK;
#pragma omp parallel
    {
        int8_t* codes = (int8_t*)malloc((size_t)H);
        float* scales = (float*)malloc(sizeof(float) * (size_t)G);
#pragma omp for schedule(static)
        for (int32_t t = 0; t < T; ++t) {
            int rc = (codes && scales) ? orc_quantize_token(x + (size_t)t * H, H, codes, scales) : ORC_ERR_ARG;
            for (int32_t j = 0; j < k && rc == ORC_OK; ++j) {
                int32_t r = slot[(size_t)t * k + j];
                if (r < 0 || r >= R) { rc = ORC_ERR_ARG; break; }
                memcpy(pool_codes + (size_t)r * H, codes, (size_t)H);
                memcpy(pool_scales + (size_t)r * G, scales, sizeof(float) * (size_t)G);
            }
            if (rc != ORC_OK) orc_note_error(t, rc, &err_t, &err_rc);
        }
        free(codes);
        free(scales);
    }
    return err_rc;
}

/* --------------------------------------------------------- experts (a9) -- */

/* Identity experts: out[r, i] = bf16( code[r, i] * scale[r, i/128] ) in fp32. */
int orc_identity_experts(const int8_t* codes, const float* scales, int32_t rows, int32_t H,
                         uint16_t* out) {
    if (!codes || !scales || !out || rows < 0 || H < 128 || H % 128 != 0) return ORC_ERR_ARG;
    const int32_t G = H / 128;
#pragma omp parallel for schedule(static)
    for (int32_t r = 0; r < rows; ++r)
        for (int32_t i = 0; i < H; ++i) {
            float v = (float)codes[(size_t)r * H + i] * scales[(size_t)r * G + i / 128];
            out[(size_t)r * H + i] = orc_f32_to_bf16(v);
        }
    return ORC_OK;
}

/* -------------------------------------------------------- combine (a10) -- */

/*
 * Gate-weighted gather-reduce back to token order.
 *   ex_out  bf16 bits [R, H]  expert outputs, one row per slot
 *   slot    int32 [T, k], gates fp32 [T, k]
 *   y       bf16 bits [T, H]
 * acc = 0; for j = 0..k-1: acc = fmaf(gate_j, ex_out[slot_j, i], acc);
 * y = bf16(acc).
 */
static int orc_combine_token(const uint16_t* ex_out, int32_t R, int32_t H, int32_t k,
                             const int32_t* slot, const float* gates, uint16_t* y) {
    for (int32_t j = 0; j < k; ++j) {
        int32_t r = slot[j];
        if (r < 0 || r >= R) return ORC_ERR_ARG;
    }
    for (int32_t i = 0; i < H; ++i) {
        float acc = 0.0f;
        for (int32_t j = 0; j < k; ++j)
            acc = fmaf(gates[j], orc_bf16_to_f32(ex_out[(size_t)slot[j] * H + i]), acc);
        y[i] = orc_f32_to_bf16(acc);
    }
    return ORC_OK;
}

int orc_combine(const uint16_t* ex_out, int32_t R, int32_t H, int32_t k,
                const int32_t* slot, const float* gates, int32_t T, uint16_t* y) {
    if (!ex_out || !slot || !gates || !y || T < 0 || k < 1 || H < 1) return ORC_ERR_ARG;
    int32_t err_t = -1;
    int err_rc = ORC_OK;
#pragma omp parallel for schedule(static)
    for (int32_t t = 0; t < T; ++t) {
        int rc = orc_combine_token(ex_out, R, H, k, slot + (size_t)t * k, gates + (size_t)t * k,
                                   y + (size_t)t * H);
        if (rc != ORC_OK) orc_note_error(t, rc, &err_t, &err_rc);
    }
    return err_rc;
}

/*
 * Combine for a subset of tokens only: rows of y for token ids tok[0..n-1].
 * Same arithmetic as orc_combine; y_sub is [n, H].  Used to check large
 * batches on sampled tokens.
 */
int orc_combine_tokens(const uint16_t* ex_out, int32_t R, int32_t H, int32_t k,
                       const int32_t* slot, const float* gates,
                       const int32_t* tok, int32_t n, uint16_t* y_sub) {
    if (!ex_out || !slot || !gates || !tok || !y_sub || n < 0 || k < 1 || H < 1) return ORC_ERR_ARG;
    int32_t err_s = -1;
    int err_rc = ORC_OK;
#pragma omp parallel for schedule(static)
    for (int32_t s = 0; s < n; ++s) {
        int32_t t = tok[s];
        int rc = orc_combine_token(ex_out, R, H, k, slot + (size_t)t * k, gates + (size_t)t * k,
                                   y_sub + (size_t)s * H);
        if (rc != ORC_OK) orc_note_error(s, rc, &err_s, &err_rc);
    }
    return err_rc;
}

/* bf16 helpers exposed for the oracle's own pin tests. */
void orc_f32_to_bf16_array(const float* in, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(in[i]);
}
