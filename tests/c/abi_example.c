/*
 * A plain C caller of the library's C ABI (include/b200norm.h): no Python,
 * no torch.  Without B200NORM_EXAMPLE_GPU it only exercises what needs no
 * GPU (version, status strings, argument errors, which are reported before
 * anything touches the device).  With it, it also runs
 * SkipSimplifiedLayerNormalization on the README usage example's closed-form
 * case: input [1, 3], skip [2, 1] -> S = [3, 4]; with gamma = 1 and eps = 0,
 * Y = S / sqrt((9 + 16) / 2) = [0.8485281374, 1.1313708499].
 * Exit status 0 on success.
 */
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "b200norm.h"

#ifdef B200NORM_EXAMPLE_GPU
#include <cuda_runtime.h>
#endif

static int fails = 0;

static void check(int ok, const char* what) {
    if (!ok) {
        fprintf(stderr, "FAIL: %s\n", what);
        ++fails;
    }
}

int main(void) {
    check(b200norm_version() == 1, "version");
    check(strcmp(b200norm_status_string(B200NORM_OK), "B200NORM_OK") == 0, "status string");
    /* hidden == 0 is an argument error, reported before any device work */
    b200norm_status st = b200norm_skip_rms(NULL, NULL, NULL, NULL, NULL, NULL, 2, 0,
                                           B200NORM_F32, 1e-5f, NULL);
    check(st == B200NORM_ERR_INVALID_ARGUMENT, "hidden = 0 rejected");
    check(strlen(b200norm_last_error()) > 0, "last_error explains it");
    st = b200norm_gated_rms(NULL, NULL, NULL, NULL, 12, 5, B200NORM_F16, 1e-5f, NULL);
    check(st == B200NORM_ERR_INVALID_ARGUMENT, "numel not a multiple of C rejected");

#ifdef B200NORM_EXAMPLE_GPU
    const float x[2] = {1.0f, 3.0f}, skip[2] = {2.0f, 1.0f}, gamma[2] = {1.0f, 1.0f};
    float y[2] = {0.0f, 0.0f}, s[2] = {0.0f, 0.0f};
    float *dx, *dskip, *dgamma, *dy, *ds;
    cudaStream_t stream;
    if (cudaStreamCreate(&stream) != cudaSuccess || cudaMalloc((void**)&dx, sizeof(x)) ||
        cudaMalloc((void**)&dskip, sizeof(skip)) || cudaMalloc((void**)&dgamma, sizeof(gamma)) ||
        cudaMalloc((void**)&dy, sizeof(y)) || cudaMalloc((void**)&ds, sizeof(s))) {
        fprintf(stderr, "FAIL: CUDA setup\n");
        return 1;  /* nothing below may run on unallocated pointers */
    }
    cudaMemcpy(dx, x, sizeof(x), cudaMemcpyHostToDevice);
    cudaMemcpy(dskip, skip, sizeof(skip), cudaMemcpyHostToDevice);
    cudaMemcpy(dgamma, gamma, sizeof(gamma), cudaMemcpyHostToDevice);
    st = b200norm_skip_rms(dx, dskip, dgamma, NULL, dy, ds, 1, 2, B200NORM_F32, 0.0f, stream);
    check(st == B200NORM_OK, "skip_rms");
    check(cudaStreamSynchronize(stream) == cudaSuccess, "sync");
    cudaMemcpy(y, dy, sizeof(y), cudaMemcpyDeviceToHost);
    cudaMemcpy(s, ds, sizeof(s), cudaMemcpyDeviceToHost);
    check(s[0] == 3.0f && s[1] == 4.0f, "S = [3, 4]");
    check(fabs(y[0] - 0.8485281374) < 1e-6 && fabs(y[1] - 1.1313708499) < 1e-6, "Y");
    cudaFree(dx);
    cudaFree(dskip);
    cudaFree(dgamma);
    cudaFree(dy);
    cudaFree(ds);
    cudaStreamDestroy(stream);
#endif
    if (fails == 0) printf("ok\n");
    return fails == 0 ? 0 : 1;
}
