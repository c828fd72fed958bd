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
#include "quant.cuh"
#include "trace.cuh"

MOE_TRACE_BUFFERS(tr_dispatch)

namespace moe {
namespace {

constexpr int kDispatchThreads = 256;  // 8 warps, 8 (token, segment) items per CTA

// X_EARLY: load and quantize x before waiting for the preceding kernel
// (moe_dispatch_after_plan); otherwise x is read after the wait, like every
// other input (moe_dispatch).
template <bool X_EARLY>
__global__ void __launch_bounds__(kDispatchThreads)
dispatch_kernel(const uint16_t* __restrict__ x, int T, int H, int k, const int32_t* __restrict__ slot,
                int8_t* __restrict__ codes, float* __restrict__ scales, int Gs, int32_t* __restrict__ err) {
    // Trace stages (warp 0 of the CTA): 0 start, 1 quantized, 2 slots read,
    // 3 stores issued.
    MOE_TRACE_SM(tr_dispatch);
    MOE_TRACE_MARK(tr_dispatch, 0);
    const int lane = threadIdx.x & 31;
    const int segs = (H + kSegElems - 1) / kSegElems;
    const long long item = (long long)blockIdx.x * (kDispatchThreads / 32) + (threadIdx.x >> 5);
    const int t = (int)(item / segs);
    const int seg = (int)(item - (long long)t * segs);
    if (t >= T) return;

    // In the X_EARLY form x is loaded and quantized before the wait.  That is
    // correct only when the kernel launched just before this one never writes
    // x and lets its dependents start only after its own wait has returned
    // (then everything earlier on the stream has completed and its writes are
    // visible): the plan kernels meet both, and moe_dispatch_after_plan makes
    // this the caller's precondition.  The default form waits first.  The
    // slots come from the plan and are always read after the wait.
    // Dependents may start only after the wait, as in every kernel of the
    // library, so that whatever runs next on the stream sees all writes made
    // before this kernel.
    if (!X_EARLY) grid_dependency_sync();
    const SegLoad ld = load_segment(x, t, H, seg, lane);
    const SegQuant qz = quantize_segment(ld);
    MOE_TRACE_MARK(tr_dispatch, 1);
    if (X_EARLY) grid_dependency_sync();
    allow_dependents();
    const int my_slot = (lane < k) ? slot[(size_t)t * k + lane] : 0;
    MOE_TRACE_MARK(tr_dispatch, 2);
    store_segment(ld, qz, my_slot, k, T * k, H, Gs, seg, codes, scales, err);
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
                            float* scales, int Gs, int32_t* err, bool x_early, cudaStream_t s, uint64_t* launches) {
    const long long items = (long long)T * ((H + kSegElems - 1) / kSegElems);
    const long long blocks = (items + (kDispatchThreads / 32) - 1) / (kDispatchThreads / 32);
    cudaError_t e = x_early ? launch_pdl(dispatch_kernel<true>, dim3((unsigned)blocks), dim3(kDispatchThreads), 0, s,
                                         x, T, H, k, slot, codes, scales, Gs, err)
                            : launch_pdl(dispatch_kernel<false>, dim3((unsigned)blocks), dim3(kDispatchThreads), 0,
                                         s, x, T, H, k, slot, codes, scales, Gs, err);
    if (e == cudaSuccess) *launches += 1;
    return e;
}

cudaError_t launch_identity_experts(const int8_t* codes, const float* scales, int rows, int H, int Gs,
                                    uint16_t* ex_out, cudaStream_t s, uint64_t* launches) {
    const long long n = (long long)rows * (H / 16);
    long long blocks = (n + kExpertThreads - 1) / kExpertThreads;
    int dev = 0, sms = 1;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long cap = 16LL * (sms > 0 ? sms : 1);  // grid-stride: 16 CTAs of 256 per SM
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaError_t e = launch_pdl(identity_experts_kernel, dim3((unsigned)blocks), dim3(kExpertThreads), 0, s, codes,
                               scales, rows, H, Gs, ex_out);
    if (e == cudaSuccess) *launches += 1;
    return e;
}

}  // namespace moe
