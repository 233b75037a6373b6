/*
 * c_abi_client.c -- a client of the C ABI with no Python and no torch: device
 * buffers from the CUDA runtime, one decode through dattn_decode_f16_ex (caller
 * workspace) and one through dattn_decode_f16 (library workspace), each
 * compared element by element with the fp64 oracle (|out - ref| <= 2e-3 +
 * 1e-2 |ref|), plus one rejected call.  Built and run by
 * tests/test_c_abi_client_gpu.py; prints "ok" and exits 0 on success.
 */
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include "dattn.h"

/* from the oracle (test infrastructure, oracle/oracle.c) */
void oracle_decode_f64(const uint16_t *Q, const uint16_t *K, const uint16_t *V, int64_t B,
                       int64_t H, int64_t D, int64_t S, const uint32_t *current_pos,
                       double *out, int nthreads);
uint16_t oracle_f32_to_f16_rne(float f);
double oracle_f16_to_f64(uint16_t h);

#define CHECK_CUDA(x)                                                              \
    do {                                                                           \
        cudaError_t e_ = (x);                                                      \
        if (e_ != cudaSuccess) {                                                   \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));               \
            return 2;                                                              \
        }                                                                          \
    } while (0)

/* 64-bit linear congruential generator (Knuth's MMIX constants) */
static uint64_t g_state = 20260002u;
static float uniform_pm2(void) {
    g_state = g_state * 6364136223846793005ULL + 1442695040888963407ULL;
    return (float)((g_state >> 11) * (1.0 / 9007199254740992.0)) * 4.0f - 2.0f;
}

static int compare(const uint16_t *got, const double *ref, size_t n, const char *what) {
    size_t bad = 0;
    double worst = 0.0;
    for (size_t i = 0; i < n; ++i) {
        const double err = fabs(oracle_f16_to_f64(got[i]) - ref[i]);
        if (!(err <= 2e-3 + 1e-2 * fabs(ref[i]))) ++bad;
        if (err > worst) worst = err;
    }
    if (bad) fprintf(stderr, "%s: %zu of %zu out of tolerance (max err %g)\n", what, bad, n, worst);
    return bad != 0;
}

int main(void) {
    const int B = 3, H = 8, D = 128, S = 1000;
    const uint32_t cp[3] = {999, 0, 517};
    const size_t nq = (size_t)B * H * D, nkv = (size_t)B * S * H * D;
    uint16_t *q = malloc(nq * 2), *k = malloc(nkv * 2), *v = malloc(nkv * 2), *got = malloc(nq * 2);
    double *ref = malloc(nq * sizeof(double));
    if (!q || !k || !v || !got || !ref) return 2;
    for (size_t i = 0; i < nq; ++i) q[i] = oracle_f32_to_f16_rne(uniform_pm2());
    for (size_t i = 0; i < nkv; ++i) k[i] = oracle_f32_to_f16_rne(uniform_pm2());
    for (size_t i = 0; i < nkv; ++i) v[i] = oracle_f32_to_f16_rne(uniform_pm2());
    oracle_decode_f64(q, k, v, B, H, D, S, cp, ref, 0);

    void *dq, *dk, *dv, *dout, *dcp, *dws;
    CHECK_CUDA(cudaMalloc(&dq, nq * 2));
    CHECK_CUDA(cudaMalloc(&dk, nkv * 2));
    CHECK_CUDA(cudaMalloc(&dv, nkv * 2));
    CHECK_CUDA(cudaMalloc(&dout, nq * 2));
    CHECK_CUDA(cudaMalloc(&dcp, sizeof cp));
    CHECK_CUDA(cudaMemcpy(dq, q, nq * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dk, k, nkv * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dv, v, nkv * 2, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dcp, cp, sizeof cp, cudaMemcpyHostToDevice));

    size_t wsb = 0;
    int st = dattn_decode_workspace_bytes(B, H, D, S, 0, &wsb);
    if (st != DATTN_OK) {
        fprintf(stderr, "workspace query: %s\n", dattn_status_string(st));
        return 1;
    }
    CHECK_CUDA(cudaMalloc(&dws, wsb > 16 ? wsb : 16));

    int fail = 0;
    st = dattn_decode_f16_ex(dq, dk, dv, dout, B, H, D, S, dcp, dws, wsb, 0, NULL);
    if (st != DATTN_OK) {
        fprintf(stderr, "dattn_decode_f16_ex: %s (%s)\n", dattn_status_string(st), dattn_last_error());
        return 1;
    }
    CHECK_CUDA(cudaMemcpy(got, dout, nq * 2, cudaMemcpyDeviceToHost));
    fail |= compare(got, ref, nq, "dattn_decode_f16_ex");

    CHECK_CUDA(cudaMemset(dout, 0, nq * 2));
    st = dattn_decode_f16(dq, dk, dv, dout, B, H, D, S, dcp, NULL);
    if (st != DATTN_OK) {
        fprintf(stderr, "dattn_decode_f16: %s (%s)\n", dattn_status_string(st), dattn_last_error());
        return 1;
    }
    CHECK_CUDA(cudaMemcpy(got, dout, nq * 2, cudaMemcpyDeviceToHost));
    fail |= compare(got, ref, nq, "dattn_decode_f16");

    /* a misaligned Q is rejected on the host, with a message */
    st = dattn_decode_f16_ex((const char *)dq + 2, dk, dv, dout, B, H, D, S, dcp, dws, wsb, 0, NULL);
    if (st != DATTN_ERR_MISALIGNED || dattn_last_error()[0] == '\0') {
        fprintf(stderr, "misaligned Q: got %s\n", dattn_status_string(st));
        fail = 1;
    }
    if (dattn_device_error(1) != DATTN_OK) {
        fprintf(stderr, "device error word set\n");
        fail = 1;
    }
    cudaFree(dq);
    cudaFree(dk);
    cudaFree(dv);
    cudaFree(dout);
    cudaFree(dcp);
    cudaFree(dws);
    free(q);
    free(k);
    free(v);
    free(got);
    free(ref);
    if (!fail) printf("ok\n");
    return fail;
}
