// dispatch.cu -- FusedDispatch data phase: per-token INT8 quantization with
// one fp32 scale per 128 elements, scattered into the token's k expert slots.
//
// CloudMatrix384 write-up, "FusedDispatch and FusedCombine": early INT8
// quantization before the data moves (14 KB bf16 -> about 7.5 KB per token
// with its scales), direct writes into pre-allocated receive buffers, and a
// token-level pipeline of load -> quantize/address -> write.
//
// GPU mapping: one warp per (token, 512-element segment).  Each lane loads 16
// bf16 values (two 16-byte loads), a group of 128 elements spans 8 lanes, so
// amax is a 3-step xor-shuffle; codes are rint((x * 127) / amax), the
// correctly rounded fp32 quotient (one reciprocal per group and Markstein's
// correction per element) and round-half-even conversion; the lane's 16 codes leave as
// one 16-byte store into each of the token's k rows; the 4 group scales of
// the segment leave as one 16-byte store per row.  Reads of x are streamed
// once; every byte of every destination row is written exactly once.
#include "moe_internal.h"
#include "ptx.cuh"
#include "trace.cuh"

MOE_TRACE_BUFFERS(tr_dispatch)

namespace moe {
namespace {

constexpr int kDispatchThreads = 256;  // 8 warps, 8 (token, segment) items per CTA
constexpr int kSegElems = 512;         // 32 lanes x 16 elements

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

__global__ void __launch_bounds__(kDispatchThreads)
dispatch_kernel(const uint16_t* __restrict__ x, int T, int H, int k, const int32_t* __restrict__ slot,
                int8_t* __restrict__ codes, float* __restrict__ scales, int Gs, int32_t* __restrict__ err) {
    // Trace stages (warp 0 of the CTA): 0 start, 1 row and slots loaded,
    // 2 quantized, 3 stores issued.
    grid_dependency_sync();
    allow_dependents();
    MOE_TRACE_SM(tr_dispatch);
    MOE_TRACE_MARK(tr_dispatch, 0);
    const int lane = threadIdx.x & 31;
    const int segs = (H + kSegElems - 1) / kSegElems;
    const long long item = (long long)blockIdx.x * (kDispatchThreads / 32) + (threadIdx.x >> 5);
    const int t = (int)(item / segs);
    const int seg = (int)(item - (long long)t * segs);
    if (t >= T) return;

    const int chunk = seg * 32 + lane;  // 16-element chunk within the row
    const bool active = chunk * 16 < H;
    const int rows = T * k;

    uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
    if (active) {
        const uint16_t* src = x + (size_t)t * H + (size_t)chunk * 16;
        lo = ld_stream16(src);
        hi = ld_stream16(src + 8);
    }
    const int my_slot = (lane < k) ? slot[(size_t)t * k + lane] : 0;

    float v[16];
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
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
    MOE_TRACE_MARK(tr_dispatch, 1);

    // amax == 0 only when the whole group is +-0: dividing by 1 keeps codes 0.
    const float den = amax > 0.0f ? amax : 1.0f;
    uint4 q;
    if (den >= 0x1p-126f && den <= 0x1p125f) {  // 1/den is a normal binary32
        const float inv = __frcp_rn(den);
        q.x = quant4<true>(v[0], v[1], v[2], v[3], den, inv);
        q.y = quant4<true>(v[4], v[5], v[6], v[7], den, inv);
        q.z = quant4<true>(v[8], v[9], v[10], v[11], den, inv);
        q.w = quant4<true>(v[12], v[13], v[14], v[15], den, inv);
    } else {
        q.x = quant4<false>(v[0], v[1], v[2], v[3], den, 0.0f);
        q.y = quant4<false>(v[4], v[5], v[6], v[7], den, 0.0f);
        q.z = quant4<false>(v[8], v[9], v[10], v[11], den, 0.0f);
        q.w = quant4<false>(v[12], v[13], v[14], v[15], den, 0.0f);
    }

    const float scale = amax / 127.0f;
    float4 sc;
    sc.x = __shfl_sync(kFull, scale, 0);
    sc.y = __shfl_sync(kFull, scale, 8);
    sc.z = __shfl_sync(kFull, scale, 16);
    sc.w = __shfl_sync(kFull, scale, 24);
    MOE_TRACE_MARK(tr_dispatch, 2);

    for (int j = 0; j < k; ++j) {
        const int r = __shfl_sync(kFull, my_slot, j);
        if (r < 0 || r >= rows) {  // warp-uniform
            if (lane == 0) set_error(err, MOE_DEVERR_SLOT);
            continue;
        }
        if (active) st16(codes + (size_t)r * H + (size_t)chunk * 16, q);
    }
    // Scales of this segment's 4 groups: one 16-byte store per destination row.
    if (lane < k && my_slot >= 0 && my_slot < rows && seg * 4 < Gs)
        *reinterpret_cast<float4*>(scales + (size_t)my_slot * Gs + seg * 4) = sc;
    MOE_TRACE_MARK(tr_dispatch, 3);
}

constexpr int kExpertThreads = 256;

// ex_out[r, i] = bf16(code[r, i] * scale[r, i / 128]); one thread per 16 codes.
__global__ void __launch_bounds__(kExpertThreads)
identity_experts_kernel(const int8_t* __restrict__ codes, const float* __restrict__ scales, int rows, int H,
                        int Gs, uint16_t* __restrict__ ex_out) {
    grid_dependency_sync();
    allow_dependents();
    const int per_row = H / 16;
    const long long n = (long long)rows * per_row;
    for (long long c = (long long)blockIdx.x * kExpertThreads + threadIdx.x; c < n;
         c += (long long)gridDim.x * kExpertThreads) {
        const int r = (int)(c / per_row);
        const int ch = (int)(c - (long long)r * per_row);
        const uint4 q = ld_stream16(codes + (size_t)r * H + (size_t)ch * 16);
        const float s = scales[(size_t)r * Gs + (ch * 16) / kGroup];
        const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float a = (float)(int8_t)(qw[i] & 0xff) * s;
            const float b = (float)(int8_t)((qw[i] >> 8) & 0xff) * s;
            const float c2 = (float)(int8_t)((qw[i] >> 16) & 0xff) * s;
            const float d = (float)(int8_t)(qw[i] >> 24) * s;
            o[2 * i] = pack_bf16x2_rn(a, b);
            o[2 * i + 1] = pack_bf16x2_rn(c2, d);
        }
        uint16_t* dst = ex_out + (size_t)r * H + (size_t)ch * 16;
        st16(dst, make_uint4(o[0], o[1], o[2], o[3]));
        st16(dst + 8, make_uint4(o[4], o[5], o[6], o[7]));
    }
}

}  // namespace

#ifdef MOE_TRACE
int trace_symbols_dispatch(void** stamps, void** sms) {
    if (cudaGetSymbolAddress(stamps, tr_dispatch_t) != cudaSuccess) return -1;
    return cudaGetSymbolAddress(sms, tr_dispatch_sm) == cudaSuccess ? 0 : -1;
}
#endif

cudaError_t launch_dispatch(const uint16_t* x, int T, int H, int k, const int32_t* slot, int8_t* codes,
                            float* scales, int Gs, int32_t* err, cudaStream_t s, uint64_t* launches) {
    const long long items = (long long)T * ((H + kSegElems - 1) / kSegElems);
    const long long blocks = (items + (kDispatchThreads / 32) - 1) / (kDispatchThreads / 32);
    cudaError_t e = launch_pdl(dispatch_kernel, dim3((unsigned)blocks), dim3(kDispatchThreads), 0, s, x, T, H, k,
                               slot, codes, scales, Gs, err);
    if (e == cudaSuccess) *launches += 1;
    return e;
}

cudaError_t launch_identity_experts(const int8_t* codes, const float* scales, int rows, int H, int Gs,
                                    uint16_t* ex_out, cudaStream_t s, uint64_t* launches) {
    const long long n = (long long)rows * (H / 16);
    long long blocks = (n + kExpertThreads - 1) / kExpertThreads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    cudaError_t e = launch_pdl(identity_experts_kernel, dim3((unsigned)blocks), dim3(kExpertThreads), 0, s, codes,
                               scales, rows, H, Gs, ex_out);
    if (e == cudaSuccess) *launches += 1;
    return e;
}

}  // namespace moe
