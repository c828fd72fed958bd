// dword.cuh -- double-word (unevaluated fp32 pair) arithmetic for the gates.
//
// A gate is exp(l_j - l_0) / sum_i exp(l_i - l_0), rounded once to fp32.
// GB300 issues fp64 at a small fraction of its fp32 rate, so the route kernel
// evaluates the gates with pairs of floats (about 48 significant bits) and
// falls back to fp64 only when the pair cannot decide the fp32 rounding
// (Ziv's rounding test).  Building blocks, all in round-to-nearest fp32 with
// explicit _rn intrinsics so that the compiler cannot contract or reorder:
//   two_sum       Knuth's 2Sum: s + e == a + b exactly
//   fast_two_sum  Dekker's Fast2Sum (|a| >= |b|): s + e == a + b exactly
//   two_prod      the FMA-based exact product: p + e == a * b exactly
//   dw_add        the accurate double-word sum analysed by Joldes, Muller and
//                 Popescu ("Tight and rigorous error bounds for basic building
//                 blocks of double-word arithmetic", ACM TOMS 44(2), 2017):
//                 relative error <= 3u^2 + 13u^3, u = 2^-24
//   dw_div        Dekker's double-word quotient ("A floating-point technique
//                 for extending the available precision", Numer. Math. 18,
//                 1971): first quotient, exact remainder terms, one correction
//   exp_dw        exp(d) for a double-word d in [-64, 0]: Cody and Waite's
//                 reduction by n ln 2 (ln 2 split in three floats), a table of
//                 exp(m / 512) (Tang's table-driven method), and the Taylor
//                 polynomial of degree 4 on |r| <= 2^-10.
#pragma once

namespace moe {
namespace dword {

struct dw {
    float h, l;
};

__device__ __forceinline__ dw two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return {s, e};
}

__device__ __forceinline__ dw fast_two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

__device__ __forceinline__ dw two_prod(float a, float b) {
    const float p = __fmul_rn(a, b);
    return {p, __fmaf_rn(a, b, -p)};
}

__device__ __forceinline__ dw dw_add(dw x, dw y) {
    const dw s = two_sum(x.h, y.h);
    const dw t = two_sum(x.l, y.l);
    const dw v = fast_two_sum(s.h, __fadd_rn(s.l, t.h));
    return fast_two_sum(v.h, __fadd_rn(t.l, v.l));
}

// x / y for y > 0.  With q = RN(xh / yh), x - q y = (xh - q yh) + xl - q yl;
// xh - RN(q yh) is exact (the two are within a factor of two), so the
// remainder is the sum of four terms each at most u |x|, added in fp32; the
// correction is that remainder over yh.  Relative error below 24 u^2.
__device__ __forceinline__ dw dw_div(dw x, dw y) {
    const float q = __fdiv_rn(x.h, y.h);
    const dw p = two_prod(q, y.h);
    const float pi = __fsub_rn(x.h, p.h);
    const float rem = __fmaf_rn(-q, y.l, __fadd_rn(__fsub_rn(pi, p.l), x.l));
    return fast_two_sum(q, __fdiv_rn(rem, y.h));
}

#include "exp_table.inc"

// Ziv's rounding test for a pair q = qh + ql (qh normal, at least 2^-102;
// |ql| <= ulp(qh) / 2) whose exact value Q satisfies |Q - q| <= eps |Q|:
// RN(Q) == qh whenever |ql| + eps |qh| stays below half the gap between qh
// and its neighbour on ql's side.  That half gap is 2^(e-24) for qh in
// [2^e, 2^(e+1)), except below an exact power of two, where it is 2^(e-25).
// The gate pipeline's bound is 2^-42.35 (exp 2^-45.5; sum 15 u^2 on top of
// that; quotient 24 u^2); the test uses eps = 2^-40.
__device__ __forceinline__ bool rounds_safely(dw q) {
    const int bits = __float_as_int(q.h);
    const int expo = bits & 0x7f800000;
    float half_gap = __int_as_float(expo - (24 << 23));
    if (q.l < 0.0f && (bits & 0x007fffff) == 0) half_gap = __fmul_rn(half_gap, 0.5f);
    return fabsf(q.l) < __fsub_rn(half_gap, __fmul_rn(q.h, 0x1p-40f));
}

// exp(d), d = dh + dl exactly, -64 <= dh <= 0.  `table` holds kExpTable
// (staged in shared memory by the caller).  Relative error below 2^-45.5:
// reduction 2^-48.4, table 2^-49.1, assembly 2^-46.1, polynomial 2^-55.
__device__ __forceinline__ dw exp_dw(float dh, float dl, const float2* table) {
    // d = n ln2 + r: n ln2A is exact (|n| <= 93 < 2^8), dh - n ln2A is exact
    // by Sterbenz's lemma, n ln2B exactly as a pair, n ln2C to 2^-58.
    const float n = rintf(__fmul_rn(dh, kInvLn2));
    const float a = __fsub_rn(dh, __fmul_rn(n, kLn2A));
    const dw b = two_prod(n, kLn2B);
    const float c = __fmul_rn(n, kLn2C);
    const dw h1 = two_sum(a, -b.h);
    const dw h2 = two_sum(h1.h, dl);
    const dw r = two_sum(h2.h, __fsub_rn(__fsub_rn(__fadd_rn(h1.l, h2.l), b.l), c));
    // r = m / 512 + r1 with |r1| <= 2^-10; r.h - m / 512 is exact.
    const float m = rintf(__fmul_rn(r.h, 512.0f));
    const dw r1 = two_sum(__fmaf_rn(-m, 1.0f / 512.0f, r.h), r.l);
    // p = r1 + r1^2 / 2 + r1^3 / 6 + r1^4 / 24 as a pair (the square exactly).
    const dw sq = two_prod(r1.h, r1.h);
    const float sq_l = __fmaf_rn(2.0f * r1.h, r1.l, sq.l);
    const float c34 = __fmul_rn(__fmul_rn(sq.h, r1.h), __fmaf_rn(r1.h, 1.0f / 24.0f, 1.0f / 6.0f));
    dw p = two_sum(r1.h, __fmul_rn(0.5f, sq.h));
    p = fast_two_sum(p.h, __fadd_rn(p.l, __fadd_rn(r1.l, __fmaf_rn(0.5f, sq_l, c34))));
    // exp(r) = T (1 + p), T = exp(m / 512) from the table.
    int idx = (int)m + kExpTableHalf;
    idx = idx < 0 ? 0 : (idx > 2 * kExpTableHalf ? 2 * kExpTableHalf : idx);
    const float2 t = table[idx];
    const dw tp = two_prod(t.x, p.h);
    const float small = __fadd_rn(tp.l, __fmaf_rn(t.x, p.l, __fmul_rn(t.y, p.h)));
    const dw s = two_sum(t.x, tp.h);
    dw e = fast_two_sum(s.h, __fadd_rn(s.l, __fadd_rn(t.y, small)));
    // times 2^n (n >= -93: the scale factor is a normal float).
    const float scale = __int_as_float((127 + (int)n) << 23);
    e.h = __fmul_rn(e.h, scale);
    e.l = __fmul_rn(e.l, scale);
    return e;
}

}  // namespace dword
}  // namespace moe
