// combine.cu -- FusedCombine: gate-weighted gather-reduce of the k bf16 expert
// rows of every token back to token order.
//
// CloudMatrix384 write-up, "FusedDispatch and FusedCombine": expert output
// return is the third exchange the fused operators absorb; combine moves bf16
// rows (14 KB per copy at hidden 7168).  The reduction is a pull: each token
// reads its own k rows (StrataCL analysis, section 3.4: data-movement
// collectives pull remote slices into the local output) and accumulates in
// fp32 with one fused multiply-add per copy, in ascending j, so the result
// does not depend on scheduling.
//
// GPU mapping: one warp per (token, 256-element segment); a lane owns one
// 8-element chunk (16 bytes) of every copy and keeps KB = min(k, 8) copies'
// 16-byte loads in flight before it accumulates them in order.  KB is a
// template parameter, so a smaller k holds fewer registers and more CTAs fit
// on an SM (k = 6: five CTAs instead of four, 3.5 % faster at hidden 2048).
#include "moe_internal.h"
#include "ptx.cuh"
#include "trace.cuh"

MOE_TRACE_BUFFERS(tr_combine)

namespace moe {
namespace {

constexpr int kCombineThreads = 256;  // 8 warps
constexpr int kChunks = 1;            // 16-byte chunks per lane per item
constexpr int kSegElems = 32 * 8 * kChunks;

template <int KB>  // copies loaded before accumulating
__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(const uint16_t* __restrict__ ex_out, const int32_t* __restrict__ slot,
               const float* __restrict__ gates, int T, int H, int k, uint16_t* __restrict__ y,
               int32_t* __restrict__ err) {
    // Trace stages (warp 0 of the CTA): 0 start, 1 slots and gates loaded,
    // 2 accumulation done, 3 output stored.
    // No early launch_dependents: the kernel after combine is normally the
    // next batch's plan, whose CTAs would sit on SMs in their wait while this
    // grid streams.  Letting dependents start only at exit measured 1 us
    // shorter per pipelined 4096-token step (124.3 vs 125.3 us).
    grid_dependency_sync();
    MOE_TRACE_SM(tr_combine);
    MOE_TRACE_MARK(tr_combine, 0);
    const int lane = threadIdx.x & 31;
    const int segs = (H + kSegElems - 1) / kSegElems;
    const long long item = (long long)blockIdx.x * (kCombineThreads / 32) + (threadIdx.x >> 5);
    const int t = (int)(item / segs);
    const int seg = (int)(item - (long long)t * segs);
    if (t >= T) return;

    const int rows = T * k;
    int my_slot = 0;
    float my_gate = 0.0f;
    if (lane < k) {
        my_slot = slot[(size_t)t * k + lane];
        my_gate = gates[(size_t)t * k + lane];
    }
    int bad = (lane < k) && (my_slot < 0 || my_slot >= rows);
    bad = __any_sync(kFull, bad);
    if (bad) {
        if (lane == 0) set_error(err, MOE_DEVERR_SLOT);
        return;
    }
    MOE_TRACE_MARK(tr_combine, 1);

    int col[kChunks];
    bool act[kChunks];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        col[c] = (seg * 32 * kChunks + c * 32 + lane) * 8;
        act[c] = col[c] < H;
    }

    float acc[kChunks][8];
#pragma unroll
    for (int c = 0; c < kChunks; ++c)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[c][e] = 0.0f;

    for (int jb = 0; jb < k; jb += KB) {
        uint4 d[KB][kChunks];
#pragma unroll
        for (int jj = 0; jj < KB; ++jj) {
            const int j = jb + jj;
            const int r = __shfl_sync(kFull, my_slot, j & 31);
#pragma unroll
            for (int c = 0; c < kChunks; ++c) {
                d[jj][c] = make_uint4(0, 0, 0, 0);
                if (j < k && act[c]) d[jj][c] = ld_stream16(ex_out + (size_t)r * H + col[c]);
            }
        }
#pragma unroll
        for (int jj = 0; jj < KB; ++jj) {
            const int j = jb + jj;
            const float g = __shfl_sync(kFull, my_gate, j & 31);
            if (j < k) {
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                    const uint32_t w[4] = {d[jj][c].x, d[jj][c].y, d[jj][c].z, d[jj][c].w};
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc[c][2 * i] = __fmaf_rn(g, bf16_lo(w[i]), acc[c][2 * i]);
                        acc[c][2 * i + 1] = __fmaf_rn(g, bf16_hi(w[i]), acc[c][2 * i + 1]);
                    }
                }
            }
        }
    }

    MOE_TRACE_MARK(tr_combine, 2);
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
        if (!act[c]) continue;
        uint4 o;
        o.x = pack_bf16x2_rn(acc[c][0], acc[c][1]);
        o.y = pack_bf16x2_rn(acc[c][2], acc[c][3]);
        o.z = pack_bf16x2_rn(acc[c][4], acc[c][5]);
        o.w = pack_bf16x2_rn(acc[c][6], acc[c][7]);
        st16(y + (size_t)t * H + col[c], o);
    }
    MOE_TRACE_MARK(tr_combine, 3);
}

}  // namespace

#ifdef MOE_TRACE
int trace_symbols_combine(void** stamps, void** sms) {
    if (cudaGetSymbolAddress(stamps, tr_combine_t) != cudaSuccess) return -1;
    return cudaGetSymbolAddress(sms, tr_combine_sm) == cudaSuccess ? 0 : -1;
}
#endif

cudaError_t launch_combine(const uint16_t* ex_out, const int32_t* slot, const float* gates, int T, int H, int k,
                           uint16_t* y, int32_t* err, cudaStream_t s, uint64_t* launches) {
    const long long items = (long long)T * ((H + kSegElems - 1) / kSegElems);
    const long long blocks = (items + (kCombineThreads / 32) - 1) / (kCombineThreads / 32);
    cudaError_t e;
#define MOE_COMBINE_CASE(KB)                                                                                    \
    e = launch_pdl(combine_kernel<KB>, dim3((unsigned)blocks), dim3(kCombineThreads), 0, s, ex_out, slot, gates, \
                   T, H, k, y, err)
    switch (k < 8 ? k : 8) {
        case 1: MOE_COMBINE_CASE(1); break;
        case 2: MOE_COMBINE_CASE(2); break;
        case 3: MOE_COMBINE_CASE(3); break;
        case 4: MOE_COMBINE_CASE(4); break;
        case 5: MOE_COMBINE_CASE(5); break;
        case 6: MOE_COMBINE_CASE(6); break;
        case 7: MOE_COMBINE_CASE(7); break;
        default: MOE_COMBINE_CASE(8); break;
    }
#undef MOE_COMBINE_CASE
    if (e == cudaSuccess) *launches += 1;
    return e;
}

}  // namespace moe
