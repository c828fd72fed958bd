/*
 * The fully fused expert-parallel split of R ranks, emulated on one GPU and
 * driven from plain C through include/moe.h, include/moe_ep.h and the CUDA
 * runtime only: every rank plans its batch in its own pool, the window starts
 * come from every rank's counts on the device, every rank's tokens are
 * quantized and written straight into the owners' receive buffers (recording
 * where each copy went), the owners' identity experts run on what they
 * received, and every rank reduces its tokens from the owners' buffers.
 * Used by tests/test_gpu_c_abi.py.
 *
 *   c_abi_ep_step <in> <out>
 *   in:  int32 R, T, H, E, P, k, has_rep; then per rank fp32 logits [T, E] and
 *        uint16 x [T, H]; if has_rep: int32 rep_off [E + 1], int32 rep_ids [P]
 *   out: per owner int32 rows received; per rank uint16 y [T, H]; int32 the
 *        OR of every pool's error word
 * Exit status 0 on success, otherwise the failing step's number.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "moe.h"
#include "moe_ep.h"

static int rd(FILE* f, void* p, size_t n) { return fread(p, 1, n, f) == n ? 0 : 1; }

int main(int argc, char** argv) {
    if (argc != 3) return 1;
    FILE* fi = fopen(argv[1], "rb");
    if (!fi) return 2;
    int32_t hdr[7];
    if (rd(fi, hdr, sizeof hdr)) return 3;
    const int32_t R = hdr[0], T = hdr[1], H = hdr[2], E = hdr[3], P = hdr[4], k = hdr[5], has_rep = hdr[6];
    if (R < 1 || R > MOE_EP_MAX_RANKS || T < 1) return 4;
    const size_t n_log = (size_t)T * E, n_x = (size_t)T * H, cap = (size_t)R * T * k;
    float* h_logits = (float*)malloc(n_log * sizeof(float) * R);
    uint16_t* h_x = (uint16_t*)malloc(n_x * sizeof(uint16_t) * R);
    int32_t* h_off = (int32_t*)malloc((size_t)(E + 1) * sizeof(int32_t));
    int32_t* h_ids = (int32_t*)malloc((size_t)P * sizeof(int32_t));
    if (!h_logits || !h_x || !h_off || !h_ids) return 5;
    for (int r = 0; r < R; ++r)
        if (rd(fi, h_logits + n_log * r, n_log * sizeof(float)) || rd(fi, h_x + n_x * r, n_x * sizeof(uint16_t)))
            return 6;
    if (has_rep && (rd(fi, h_off, (size_t)(E + 1) * 4) || rd(fi, h_ids, (size_t)P * 4))) return 7;
    fclose(fi);

    moe_desc d;
    d.T_max = T; d.H = H; d.E = E; d.P = P; d.k = k; d.group = 128; d.n_sets = 1;
    size_t ws_bytes = 0;
    if (moe_pool_bytes(&d, &ws_bytes) != MOE_OK) return 10;
    cudaStream_t s;
    if (cudaStreamCreate(&s) != cudaSuccess) return 11;
    void *d_off = NULL, *d_ids = NULL, *d_start = NULL, *d_rows = NULL;
    if (cudaMalloc(&d_off, (size_t)(E + 1) * 4) != cudaSuccess || cudaMalloc(&d_ids, (size_t)P * 4) != cudaSuccess ||
        cudaMalloc(&d_start, (size_t)R * P * 4) != cudaSuccess || cudaMalloc(&d_rows, (size_t)R * 4) != cudaSuccess)
        return 12;
    if (has_rep && (cudaMemcpyAsync(d_off, h_off, (size_t)(E + 1) * 4, cudaMemcpyHostToDevice, s) != cudaSuccess ||
                    cudaMemcpyAsync(d_ids, h_ids, (size_t)P * 4, cudaMemcpyHostToDevice, s) != cudaSuccess))
        return 13;

    /* Per rank: its pool, inputs, output and copy record; per owner: its
     * receive buffers (worst case: every rank's every copy). */
    moe_pool* pool[MOE_EP_MAX_RANKS];
    void *ws[MOE_EP_MAX_RANKS], *lg[MOE_EP_MAX_RANKS], *x[MOE_EP_MAX_RANKS], *y[MOE_EP_MAX_RANKS];
    int64_t* copy_row[MOE_EP_MAX_RANKS];
    int8_t* codes[MOE_EP_MAX_RANKS];
    float* scales[MOE_EP_MAX_RANKS];
    uint16_t* ex[MOE_EP_MAX_RANKS];
    const int32_t* counts[MOE_EP_MAX_RANKS];
    int64_t cap_rows[MOE_EP_MAX_RANKS];
    int32_t Gs = 0;
    for (int r = 0; r < R; ++r) {
        if (cudaMalloc(&ws[r], ws_bytes) != cudaSuccess || cudaMalloc(&lg[r], n_log * 4) != cudaSuccess ||
            cudaMalloc(&x[r], n_x * 2) != cudaSuccess || cudaMalloc(&y[r], n_x * 2) != cudaSuccess ||
            cudaMalloc((void**)&copy_row[r], (size_t)T * k * 8) != cudaSuccess)
            return 14;
        if (moe_pool_init(&d, ws[r], ws_bytes, &pool[r]) != MOE_OK) return 15;
        moe_view v;
        if (moe_pool_view(pool[r], 0, &v) != MOE_OK) return 16;
        counts[r] = v.counts;
        Gs = v.scale_stride;
        if (cudaMemcpyAsync(lg[r], h_logits + n_log * r, n_log * 4, cudaMemcpyHostToDevice, s) != cudaSuccess ||
            cudaMemcpyAsync(x[r], h_x + n_x * r, n_x * 2, cudaMemcpyHostToDevice, s) != cudaSuccess)
            return 17;
    }
    for (int q = 0; q < R; ++q) {
        if (cudaMalloc((void**)&codes[q], cap * H) != cudaSuccess ||
            cudaMalloc((void**)&scales[q], cap * Gs * 4) != cudaSuccess ||
            cudaMalloc((void**)&ex[q], cap * H * 2) != cudaSuccess)
            return 18;
        cap_rows[q] = (int64_t)cap;
    }

    for (int r = 0; r < R; ++r)
        if (moe_plan(pool[r], (const float*)lg[r], T, has_rep ? (const int32_t*)d_off : NULL,
                     has_rep ? (const int32_t*)d_ids : NULL, 0, s) != MOE_OK)
            return 20;
    if (moe_ep_recv_start_device(R, P, counts, (int32_t*)d_start, (int32_t*)d_rows, s) != MOE_OK) return 21;
    for (int r = 0; r < R; ++r)
        if (moe_ep_dispatch(pool[r], (const uint16_t*)x[r], T, 0, R, codes, scales, cap_rows,
                            (const int32_t*)d_start + (size_t)r * P, copy_row[r], s) != MOE_OK)
            return 22;
    int32_t h_rows[MOE_EP_MAX_RANKS];
    if (cudaMemcpyAsync(h_rows, d_rows, (size_t)R * 4, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return 23;
    for (int q = 0; q < R; ++q)
        if (h_rows[q] > 0 && moe_dequant_rows(codes[q], scales[q], h_rows[q], H, Gs, ex[q], s) != MOE_OK) return 24;
    const uint16_t* const* ex_c = (const uint16_t* const*)ex;
    for (int r = 0; r < R; ++r)
        if (moe_ep_combine(pool[r], T, 0, R, ex_c, cap_rows, NULL, copy_row[r], (uint16_t*)y[r], s) != MOE_OK)
            return 25;

    int32_t err_all = 0;
    for (int r = 0; r < R; ++r) {
        int32_t err = -1;
        if (moe_pool_check(pool[r], s, &err) != MOE_OK) return 26;
        err_all |= err;
    }
    FILE* fo = fopen(argv[2], "wb");
    if (!fo) return 30;
    if (fwrite(h_rows, 4, (size_t)R, fo) != (size_t)R) return 31;
    uint16_t* h_y = (uint16_t*)malloc(n_x * 2);
    if (!h_y) return 32;
    for (int r = 0; r < R; ++r) {
        if (cudaMemcpy(h_y, y[r], n_x * 2, cudaMemcpyDeviceToHost) != cudaSuccess) return 33;
        if (fwrite(h_y, 2, n_x, fo) != n_x) return 34;
    }
    if (fwrite(&err_all, 4, 1, fo) != 1) return 35;
    fclose(fo);

    for (int r = 0; r < R; ++r) {
        moe_pool_destroy(pool[r]);
        cudaFree(ws[r]); cudaFree(lg[r]); cudaFree(x[r]); cudaFree(y[r]); cudaFree(copy_row[r]);
    }
    for (int q = 0; q < R; ++q) {
        cudaFree(codes[q]); cudaFree(scales[q]); cudaFree(ex[q]);
    }
    cudaFree(d_off); cudaFree(d_ids); cudaFree(d_start); cudaFree(d_rows);
    cudaStreamDestroy(s);
    free(h_logits); free(h_x); free(h_off); free(h_ids); free(h_y);
    return 0;
}
