// quant.cuh -- the dispatch data step for one warp and one 512-element
// segment of a token row: load, per-128 INT8 quantization, scatter.
//
// CloudMatrix384 write-up, "FusedDispatch and FusedCombine": early INT8
// quantization (per token; here one fp32 scale per 128 elements) and direct
// writes into the per-expert receive buffers.
#pragma once

#include <cstdint>

#include "moe.h"
#include "ptx.cuh"

namespace moe {

constexpr int kSegElems = 512;  // 32 lanes x 16 elements

// Correctly rounded binary32 quotient a / d for d > 0 with y = RN(1/d),
// by Markstein's correction step (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990): q0 = RN(a * y) is within one ulp of a/d, the residual a - d*q0 is
// exact in one fma, and RN(q0 + r*y) is the correctly rounded quotient.
// Valid while 1/d is a normal number and nothing overflows; the caller falls
// back to the IEEE division otherwise.  Checked exhaustively against the
// IEEE division over every bf16 activation and every bf16 significand of the
// group maximum.
__device__ __forceinline__ float div_rn(float a, float d, float y) {
    const float q0 = __fmul_rn(a, y);
    const float r = __fmaf_rn(-q0, d, a);
    return __fmaf_rn(r, y, q0);
}

// Four codes rint((v * 127) / amax) packed little-endian into one word.
template <bool FAST>
__device__ __forceinline__ uint32_t quant4(float a, float b, float c, float d, float den, float inv) {
    float qa, qb, qc, qd;
    if (FAST) {
        qa = div_rn(a * 127.0f, den, inv);
        qb = div_rn(b * 127.0f, den, inv);
        qc = div_rn(c * 127.0f, den, inv);
        qd = div_rn(d * 127.0f, den, inv);
    } else {
        qa = (a * 127.0f) / den;
        qb = (b * 127.0f) / den;
        qc = (c * 127.0f) / den;
        qd = (d * 127.0f) / den;
    }
    return (uint32_t)(__float2int_rn(qa) & 0xff) | ((uint32_t)(__float2int_rn(qb) & 0xff) << 8) |
           ((uint32_t)(__float2int_rn(qc) & 0xff) << 16) | ((uint32_t)(__float2int_rn(qd) & 0xff) << 24);
}

// One lane's share of a segment: 16 elements (two 16-byte loads).
struct SegLoad {
    uint4 lo, hi;
    int chunk;    // 16-element chunk index within the row
    bool active;  // chunk lies inside the row
};

__device__ __forceinline__ SegLoad load_segment(const uint16_t* __restrict__ x, int t, int H, int seg, int lane) {
    SegLoad s;
    s.chunk = seg * 32 + lane;
    s.active = s.chunk * 16 < H;
    s.lo = make_uint4(0, 0, 0, 0);
    s.hi = make_uint4(0, 0, 0, 0);
    if (s.active) {
        const uint16_t* src = x + (size_t)t * H + (size_t)s.chunk * 16;
        s.lo = ld_stream16(src);
        s.hi = ld_stream16(src + 8);
    }
    return s;
}

// The lane's 16 codes and, in every lane, the segment's 4 group scales.
struct SegQuant {
    uint4 q;
    float4 sc;
};

// Warp-collective (all 32 lanes): a group of 128 elements spans 8 lanes, so
// amax is a 3-step xor-shuffle; scale = amax / 127; code = rint of the
// correctly rounded (x * 127) / amax, half-even; amax = 0 gives scale 0 and
// codes 0.
__device__ __forceinline__ SegQuant quantize_segment(const SegLoad& s) {
    float v[16];
    const uint32_t w[8] = {s.lo.x, s.lo.y, s.lo.z, s.lo.w, s.hi.x, s.hi.y, s.hi.z, s.hi.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[2 * i] = bf16_lo(w[i]);
        v[2 * i + 1] = bf16_hi(w[i]);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 4));

    // amax == 0 only when the whole group is +-0: dividing by 1 keeps codes 0.
    const float den = amax > 0.0f ? amax : 1.0f;
    SegQuant r;
    if (den >= 0x1p-126f && den <= 0x1p125f) {  // 1/den is a normal binary32
        const float inv = __frcp_rn(den);
        r.q.x = quant4<true>(v[0], v[1], v[2], v[3], den, inv);
        r.q.y = quant4<true>(v[4], v[5], v[6], v[7], den, inv);
        r.q.z = quant4<true>(v[8], v[9], v[10], v[11], den, inv);
        r.q.w = quant4<true>(v[12], v[13], v[14], v[15], den, inv);
    } else {
        r.q.x = quant4<false>(v[0], v[1], v[2], v[3], den, 0.0f);
        r.q.y = quant4<false>(v[4], v[5], v[6], v[7], den, 0.0f);
        r.q.z = quant4<false>(v[8], v[9], v[10], v[11], den, 0.0f);
        r.q.w = quant4<false>(v[12], v[13], v[14], v[15], den, 0.0f);
    }
    const float scale = amax / 127.0f;
    r.sc.x = __shfl_sync(kFull, scale, 0);
    r.sc.y = __shfl_sync(kFull, scale, 8);
    r.sc.z = __shfl_sync(kFull, scale, 16);
    r.sc.w = __shfl_sync(kFull, scale, 24);
    return r;
}

// Warp-collective: write the segment into each of the token's k rows
// (my_slot = slot[t, lane] in lanes < k): one 16-byte code store per lane and
// row, and the 4 group scales as one 16-byte store per row.  A slot outside
// [0, rows) is skipped and reported.
__device__ __forceinline__ void store_segment(const SegLoad& s, const SegQuant& qz, int my_slot, int k, int rows,
                                              int H, int Gs, int seg, int8_t* __restrict__ codes,
                                              float* __restrict__ scales, int32_t* __restrict__ err) {
    const int lane = threadIdx.x & 31;
    for (int j = 0; j < k; ++j) {
        const int r = __shfl_sync(kFull, my_slot, j);
        if (r < 0 || r >= rows) {  // warp-uniform
            if (lane == 0) set_error(err, MOE_DEVERR_SLOT);
            continue;
        }
        if (s.active) st16(codes + (size_t)r * H + (size_t)s.chunk * 16, qz.q);
    }
    if (lane < k && my_slot >= 0 && my_slot < rows && seg * 4 < Gs)
        *reinterpret_cast<float4*>(scales + (size_t)my_slot * Gs + seg * 4) = qz.sc;
}

}  // namespace moe
