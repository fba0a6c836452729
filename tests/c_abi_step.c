/* A plain C99 caller of the library's compute path: the caller allocates
 * every device buffer with the CUDA runtime, fills them from the host, runs
 * three fused steps (zero3_step, the persistent group included) on one
 * stream and writes the results to a file for the test to compare with the
 * oracle.  Inputs are dyadic values that binary32 and bf16 hold exactly, so
 * the test rebuilds them bit for bit:
 *   flat master f           = ((f mod 2001) - 1000) / 1024
 *   persistent master j     = ((j mod 301) - 150) / 512
 *   flat gradient (rank q)  = (((3f + 5q) mod 41) - 20) / 256
 *   persistent grad (q)     = (((7j + 3q) mod 29) - 14) / 128
 * Output file: every rank's master shard (fp32, S each), the full bf16
 * buffer (psi_pad), the persistent master (fp32) and parameters (bf16).
 * Usage: c_abi_step <output path>.  Exit 0 on success, 1 with a message. */
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "zero3.h"

#define NR 3

static int fail(const char* what) {
    printf("FAILED: %s\n", what);
    return 1;
}

static uint16_t bf16_of_exact(float x) {  /* x holds at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &x, 4);
    return (uint16_t)(u >> 16);
}

int main(int argc, char** argv) {
    if (argc != 2) return fail("usage: c_abi_step <output path>");
    const int64_t numels[4] = {3000, 10, 5000, 37};
    zero3_plan* plan = NULL;
    if (zero3_partition(numels, NULL, 4, NR, 100, 500000000, &plan) != ZERO3_OK) return fail("partition");
    zero3_plan_info info;
    if (zero3_plan_info_get(plan, &info) != ZERO3_OK) return fail("plan info");
    const int64_t S = info.shard_len, P = info.psi_pad, PP = info.psi_p, PS = info.psi_s;

    float* h_master = (float*)calloc((size_t)P, sizeof(float));
    float* h_pmaster = (float*)calloc((size_t)PS, sizeof(float));
    uint16_t* h_g = (uint16_t*)calloc((size_t)P, sizeof(uint16_t));
    uint16_t* h_pg = (uint16_t*)calloc((size_t)PS, sizeof(uint16_t));
    if (!h_master || !h_pmaster || !h_g || !h_pg) return fail("host allocation");
    for (int64_t f = 0; f < PP; ++f) h_master[f] = (float)((f % 2001) - 1000) / 1024.0f;
    for (int64_t j = 0; j < PS; ++j) h_pmaster[j] = (float)((j % 301) - 150) / 512.0f;

    void* grads[NR];
    void* pgrads[NR];
    void* master[NR];
    void* m[NR];
    void* v[NR];
    void* sparam[NR];
    void *full = NULL, *pm_master = NULL, *pm_m = NULL, *pm_v = NULL, *pm_param = NULL;
    cudaStream_t stream;
    if (cudaStreamCreate(&stream) != cudaSuccess) return fail("stream");
    for (int q = 0; q < NR; ++q) {
        if (cudaMalloc(&grads[q], (size_t)P * 2) != cudaSuccess ||
            cudaMalloc(&pgrads[q], (size_t)PS * 2 + 16) != cudaSuccess ||
            cudaMalloc(&master[q], (size_t)S * 4) != cudaSuccess ||
            cudaMalloc(&m[q], (size_t)S * 4) != cudaSuccess ||
            cudaMalloc(&v[q], (size_t)S * 4) != cudaSuccess ||
            cudaMalloc(&sparam[q], (size_t)S * 2) != cudaSuccess)
            return fail("device allocation");
        for (int64_t f = 0; f < P; ++f)
            h_g[f] = f < PP ? bf16_of_exact((float)(((3 * f + 5 * q) % 41) - 20) / 256.0f) : 0;
        for (int64_t j = 0; j < PS; ++j)
            h_pg[j] = bf16_of_exact((float)(((7 * j + 3 * q) % 29) - 14) / 128.0f);
        if (cudaMemcpy(grads[q], h_g, (size_t)P * 2, cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemcpy(pgrads[q], h_pg, (size_t)PS * 2, cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemcpy(master[q], h_master + q * S, (size_t)S * 4, cudaMemcpyHostToDevice) !=
                cudaSuccess ||
            cudaMemset(m[q], 0, (size_t)S * 4) != cudaSuccess ||
            cudaMemset(v[q], 0, (size_t)S * 4) != cudaSuccess)
            return fail("device upload");
    }
    if (cudaMalloc(&full, (size_t)P * 2) != cudaSuccess ||
        cudaMalloc(&pm_master, (size_t)PS * 4) != cudaSuccess ||
        cudaMalloc(&pm_m, (size_t)PS * 4) != cudaSuccess ||
        cudaMalloc(&pm_v, (size_t)PS * 4) != cudaSuccess ||
        cudaMalloc(&pm_param, (size_t)PS * 2) != cudaSuccess)
        return fail("device allocation");
    if (cudaMemcpy(pm_master, h_pmaster, (size_t)PS * 4, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(pm_m, 0, (size_t)PS * 4) != cudaSuccess ||
        cudaMemset(pm_v, 0, (size_t)PS * 4) != cudaSuccess)
        return fail("device upload");

    const zero3_adamw_hparams hp = {5e-5, 0.9, 0.999, 1e-8, 0.01};
    zero3_persist_state ps;
    ps.grads = (const uint16_t* const*)pgrads;
    ps.master = (float*)pm_master;
    ps.m = (float*)pm_m;
    ps.v = (float*)pm_v;
    ps.param = (uint16_t*)pm_param;
    for (int64_t t = 1; t <= 3; ++t) {
        const zero3_status st = zero3_step(
            plan, &hp, t, (const uint16_t* const*)grads, 0, (float* const*)master,
            (float* const*)m, (float* const*)v, (uint16_t* const*)sparam, (uint16_t*)full, &ps,
            0, P, (zero3_stream)stream);
        if (st != ZERO3_OK) {
            printf("FAILED: zero3_step: %s\n", zero3_status_string(st));
            return 1;
        }
    }
    if (zero3_sync((zero3_stream)stream) != ZERO3_OK) return fail("sync");

    FILE* out = fopen(argv[1], "wb");
    if (!out) return fail("open output");
    float* hf = (float*)malloc((size_t)(S > PS ? S : PS) * 4);
    uint16_t* hb = (uint16_t*)malloc((size_t)(P > PS ? P : PS) * 2);
    if (!hf || !hb) return fail("host allocation");
    for (int q = 0; q < NR; ++q) {
        if (cudaMemcpy(hf, master[q], (size_t)S * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
            return fail("read back");
        fwrite(hf, 4, (size_t)S, out);
    }
    if (cudaMemcpy(hb, full, (size_t)P * 2, cudaMemcpyDeviceToHost) != cudaSuccess)
        return fail("read back");
    fwrite(hb, 2, (size_t)P, out);
    if (cudaMemcpy(hf, pm_master, (size_t)PS * 4, cudaMemcpyDeviceToHost) != cudaSuccess)
        return fail("read back");
    fwrite(hf, 4, (size_t)PS, out);
    if (cudaMemcpy(hb, pm_param, (size_t)PS * 2, cudaMemcpyDeviceToHost) != cudaSuccess)
        return fail("read back");
    fwrite(hb, 2, (size_t)PS, out);
    if (fclose(out) != 0) return fail("write output");
    zero3_plan_destroy(plan);
    printf("ok\n");
    return 0;
}
