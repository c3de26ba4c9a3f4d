/* A plain C program that runs the forward and backward through include/adaln.h
 * on the GPU: device memory from the CUDA runtime, the library's calls on the
 * default stream, and a check of the forward's y, mean and rstd and of the
 * backward's d_shift against sums written out here in double precision.
 * fp32 I/O, B = 2, N = 64, D = 256. */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>

#include <cuda_runtime_api.h>

#include "adaln.h"

#define B 2
#define N 64
#define D 256
#define ROWS (B * N)

static int fail(const char *what) {
    printf("FAIL %s\n", what);
    return 1;
}

/* a fixed pseudo-random sequence in [-1, 1) */
static uint32_t state = 12345u;
static float next_value(void) {
    state = state * 1664525u + 1013904223u;
    return (float)((state >> 8) & 0xffffff) / 8388608.0f - 1.0f;
}

int main(void) {
    static float x[ROWS * D], dy[ROWS * D], shift[B * D], scale[B * D];
    static float y[ROWS * D], mean[ROWS], rstd[ROWS], d_shift[B * D];
    for (int i = 0; i < ROWS * D; ++i) x[i] = next_value();
    for (int i = 0; i < ROWS * D; ++i) dy[i] = next_value();
    for (int i = 0; i < B * D; ++i) shift[i] = 0.1f * next_value();
    for (int i = 0; i < B * D; ++i) scale[i] = 0.1f * next_value();

    float *dx_, *dy_, *dshift_, *dscale_, *dy_out, *dmean, *drstd, *ddx, *dds, *ddsh;
    const size_t act = sizeof(float) * ROWS * D, mod = sizeof(float) * B * D;
    if (cudaMalloc((void **)&dx_, act) || cudaMalloc((void **)&dy_, act) ||
        cudaMalloc((void **)&dshift_, mod) || cudaMalloc((void **)&dscale_, mod) ||
        cudaMalloc((void **)&dy_out, act) || cudaMalloc((void **)&dmean, sizeof(float) * ROWS) ||
        cudaMalloc((void **)&drstd, sizeof(float) * ROWS) || cudaMalloc((void **)&ddx, act) ||
        cudaMalloc((void **)&dds, mod) || cudaMalloc((void **)&ddsh, mod))
        return fail("cudaMalloc");
    cudaMemcpy(dx_, x, act, cudaMemcpyHostToDevice);
    cudaMemcpy(dy_, dy, act, cudaMemcpyHostToDevice);
    cudaMemcpy(dshift_, shift, mod, cudaMemcpyHostToDevice);
    cudaMemcpy(dscale_, scale, mod, cudaMemcpyHostToDevice);

    if (adaln_fwd(dx_, dshift_, dscale_, dy_out, dmean, drstd, B, N, D, 1e-6f, ADALN_F32, 0) !=
        ADALN_OK)
        return fail("adaln_fwd");
    const size_t ws_bytes = adaln_bwd_workspace_size(B, N, D, ADALN_F32);
    void *ws = NULL;
    if (ws_bytes == 0 || cudaMalloc(&ws, ws_bytes)) return fail("workspace");
    if (adaln_bwd(dx_, dmean, drstd, dscale_, dy_, ddx, dds, ddsh, ws, ws_bytes, B, N, D,
                  ADALN_F32, 0) != ADALN_OK)
        return fail("adaln_bwd");
    if (cudaDeviceSynchronize() != cudaSuccess) return fail("synchronize");
    cudaMemcpy(y, dy_out, act, cudaMemcpyDeviceToHost);
    cudaMemcpy(mean, dmean, sizeof(float) * ROWS, cudaMemcpyDeviceToHost);
    cudaMemcpy(rstd, drstd, sizeof(float) * ROWS, cudaMemcpyDeviceToHost);
    cudaMemcpy(d_shift, ddsh, mod, cudaMemcpyDeviceToHost);

    double worst_y = 0.0, worst_stat = 0.0, worst_dshift = 0.0;
    for (int r = 0; r < ROWS; ++r) {
        const int b = r / N;
        double m = 0.0, v = 0.0;
        for (int d = 0; d < D; ++d) m += x[r * D + d];
        m /= D;
        for (int d = 0; d < D; ++d) v += (x[r * D + d] - m) * (x[r * D + d] - m);
        v /= D;
        const double rs = 1.0 / sqrt(v + (double)1e-6f);
        worst_stat = fmax(worst_stat, fabs(mean[r] - m) + fabs(rstd[r] - rs) / rs);
        for (int d = 0; d < D; ++d) {
            const double ref = (x[r * D + d] - m) * rs * (1.0 + scale[b * D + d]) + shift[b * D + d];
            worst_y = fmax(worst_y, fabs(y[r * D + d] - ref));
        }
    }
    for (int b = 0; b < B; ++b)
        for (int d = 0; d < D; ++d) {
            double s = 0.0;
            for (int n = 0; n < N; ++n) s += dy[(b * N + n) * D + d];
            worst_dshift = fmax(worst_dshift, fabs(d_shift[b * D + d] - s));
        }
    printf("max |y - ref| %.3e, stats %.3e, max |d_shift - ref| %.3e\n", worst_y, worst_stat,
           worst_dshift);
    if (!(worst_y <= 1e-5 && worst_stat <= 1e-6 && worst_dshift <= 1e-4)) return fail("tolerance");
    printf("0 failure(s)\n");
    return 0;
}
