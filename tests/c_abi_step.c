/*
 * One whole step driven from plain C through include/moe.h and the CUDA
 * runtime only (no Python, no torch): the caller allocates the workspace and
 * its own buffers, plans, dispatches, runs the identity-expert stand-in,
 * combines, and reads results back.  Used by tests/test_gpu_c_abi.py.
 *
 *   c_abi_step <in> <out>
 *   in:  int32 T, H, E, P, k, has_rep; fp32 logits [T, E]; uint16 x [T, H];
 *        if has_rep: int32 rep_off [E + 1], int32 rep_ids [P]
 *   out: int32 slot [T, k]; uint16 y [T, H]; int32 error word
 * Exit status 0 on success, otherwise the failing step's number.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime.h>

#include "moe.h"

static int rd(FILE* f, void* p, size_t n) { return fread(p, 1, n, f) == n ? 0 : 1; }

int main(int argc, char** argv) {
    if (argc != 3) return 1;
    FILE* fi = fopen(argv[1], "rb");
    if (!fi) return 2;
    int32_t hdr[6];
    if (rd(fi, hdr, sizeof hdr)) return 3;
    const int32_t T = hdr[0], H = hdr[1], E = hdr[2], P = hdr[3], k = hdr[4], has_rep = hdr[5];
    const size_t n_log = (size_t)T * E, n_x = (size_t)T * H;
    float* h_logits = (float*)malloc(n_log * sizeof(float));
    uint16_t* h_x = (uint16_t*)malloc(n_x * sizeof(uint16_t));
    int32_t* h_off = (int32_t*)malloc((size_t)(E + 1) * sizeof(int32_t));
    int32_t* h_ids = (int32_t*)malloc((size_t)P * sizeof(int32_t));
    if (!h_logits || !h_x || !h_off || !h_ids) return 4;
    if (rd(fi, h_logits, n_log * sizeof(float)) || rd(fi, h_x, n_x * sizeof(uint16_t))) return 5;
    if (has_rep && (rd(fi, h_off, (size_t)(E + 1) * 4) || rd(fi, h_ids, (size_t)P * 4))) return 6;
    fclose(fi);

    /* The caller owns every device allocation; the library carves the pool. */
    moe_desc d;
    d.T_max = T; d.H = H; d.E = E; d.P = P; d.k = k; d.group = 128; d.n_sets = 1;
    size_t ws_bytes = 0;
    if (moe_pool_bytes(&d, &ws_bytes) != MOE_OK) return 10;
    void *ws = NULL, *d_logits = NULL, *d_x = NULL, *d_y = NULL, *d_off = NULL, *d_ids = NULL;
    if (cudaMalloc(&ws, ws_bytes) != cudaSuccess || cudaMalloc(&d_logits, n_log * 4) != cudaSuccess ||
        cudaMalloc(&d_x, n_x * 2) != cudaSuccess || cudaMalloc(&d_y, n_x * 2) != cudaSuccess ||
        cudaMalloc(&d_off, (size_t)(E + 1) * 4) != cudaSuccess || cudaMalloc(&d_ids, (size_t)P * 4) != cudaSuccess)
        return 11;
    moe_pool* pool = NULL;
    if (moe_pool_init(&d, ws, ws_bytes, &pool) != MOE_OK) return 12;
    cudaStream_t s;
    if (cudaStreamCreate(&s) != cudaSuccess) return 13;
    if (cudaMemcpyAsync(d_logits, h_logits, n_log * 4, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(d_x, h_x, n_x * 2, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return 14;
    if (has_rep && (cudaMemcpyAsync(d_off, h_off, (size_t)(E + 1) * 4, cudaMemcpyHostToDevice, s) != cudaSuccess ||
                    cudaMemcpyAsync(d_ids, h_ids, (size_t)P * 4, cudaMemcpyHostToDevice, s) != cudaSuccess))
        return 15;

    if (moe_plan(pool, (const float*)d_logits, T, has_rep ? (const int32_t*)d_off : NULL,
                 has_rep ? (const int32_t*)d_ids : NULL, 0, s) != MOE_OK)
        return 20;
    if (moe_dispatch(pool, (const uint16_t*)d_x, T, 0, s) != MOE_OK) return 21;
    if (moe_identity_experts(pool, T, 0, s) != MOE_OK) return 22;
    if (moe_combine(pool, NULL, (uint16_t*)d_y, T, 0, s) != MOE_OK) return 23;

    int32_t err = -1;
    if (moe_pool_check(pool, s, &err) != MOE_OK) return 24;
    moe_view v;
    if (moe_pool_view(pool, 0, &v) != MOE_OK) return 25;
    int32_t* h_slot = (int32_t*)malloc((size_t)T * k * 4);
    uint16_t* h_y = (uint16_t*)malloc(n_x * 2);
    if (!h_slot || !h_y) return 26;
    if (cudaMemcpy(h_slot, v.slot, (size_t)T * k * 4, cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemcpy(h_y, d_y, n_x * 2, cudaMemcpyDeviceToHost) != cudaSuccess)
        return 27;

    FILE* fo = fopen(argv[2], "wb");
    if (!fo) return 30;
    if (fwrite(h_slot, 4, (size_t)T * k, fo) != (size_t)T * k || fwrite(h_y, 2, n_x, fo) != n_x ||
        fwrite(&err, 4, 1, fo) != 1)
        return 31;
    fclose(fo);

    moe_pool_destroy(pool);
    cudaStreamDestroy(s);
    cudaFree(ws); cudaFree(d_logits); cudaFree(d_x); cudaFree(d_y); cudaFree(d_off); cudaFree(d_ids);
    free(h_logits); free(h_x); free(h_off); free(h_ids); free(h_slot); free(h_y);
    return 0;
}
