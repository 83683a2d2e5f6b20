/*
 * A plain C caller of the library's C ABI (include/b200norm.h): no Python,
 * no torch.  Without B200NORM_EXAMPLE_GPU it only exercises what needs no
 * GPU (version, status strings, argument errors, which are reported before
 * anything touches the device).  With it, it also runs each operator on a
 * closed-form case built on the README usage examples' shapes:
 *
 *   SkipSimplifiedLayerNormalization: input [1, 3], skip [2, 1] -> S = [3, 4];
 *     with gamma = 1 and eps = 0, Y = S / sqrt((9 + 16) / 2)
 *     = [0.8485281374, 1.1313708499].
 *   GatedRMSNorm, X and gate (3, 4), scale (1) (C = 1): with eps = 0 every
 *     span normalises to sign(x), so Y = sign(x) * scale * silu(g), and
 *     silu(ln 3) = (3/4) ln 3, silu(-ln 3) = -(1/4) ln 3, silu(0) = 0.
 *   SkipGroupNorm, X (2, 3, 2, 8) NHWC, skip (2, 8), 2 groups: X is a +-1
 *     checkerboard and skip is constant over each group's channels, so each
 *     group has variance 1 and S - mean = X; with eps = 0,
 *     Y = gamma[c] * X + beta[c].  Run through b200norm_skip_group with a
 *     workspace of b200norm_skip_group_workspace_size() bytes zeroed by
 *     b200norm_workspace_init(), and through b200norm_skip_group_noalloc.
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

#ifdef B200NORM_EXAMPLE_GPU
/* GatedRMSNorm with C = 1 (the usage example's shapes). */
static int gated_case(cudaStream_t stream) {
    const float L3 = 1.0986122886681098f; /* ln 3 */
    const float x[12] = {2, -3, 0.5f, 7, -1, 4, -2.5f, 1, 3, -6, 8, -0.25f};
    const float g[12] = {L3, L3, 0, -L3, L3, -L3, 0, L3, -L3, L3, 0, -L3};
    const float scale[1] = {2.0f};
    float y[12];
    float *dx, *dg, *ds, *dy;
    int bad = 0;
    if (cudaMalloc((void**)&dx, sizeof(x)) || cudaMalloc((void**)&dg, sizeof(g)) ||
        cudaMalloc((void**)&ds, sizeof(scale)) || cudaMalloc((void**)&dy, sizeof(y))) {
        fprintf(stderr, "FAIL: CUDA setup (gated)\n");
        return 1;
    }
    cudaMemcpy(dx, x, sizeof(x), cudaMemcpyHostToDevice);
    cudaMemcpy(dg, g, sizeof(g), cudaMemcpyHostToDevice);
    cudaMemcpy(ds, scale, sizeof(scale), cudaMemcpyHostToDevice);
    if (b200norm_gated_rms(dx, dg, ds, dy, 12, 1, B200NORM_F32, 0.0f, stream) != B200NORM_OK ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        fprintf(stderr, "FAIL: gated_rms call: %s\n", b200norm_last_error());
        bad = 1;
    } else {
        cudaMemcpy(y, dy, sizeof(y), cudaMemcpyDeviceToHost);
        for (int i = 0; i < 12; ++i) {
            const double silu = g[i] == 0 ? 0.0 : (g[i] > 0 ? 0.75 * L3 : -0.25 * L3);
            const double want = (x[i] > 0 ? 1.0 : -1.0) * scale[0] * silu;
            if (fabs(y[i] - want) > 1e-6 * (1.0 + fabs(want))) {
                fprintf(stderr, "FAIL: gated y[%d] = %.9g, want %.9g\n", i, y[i], want);
                bad = 1;
            }
        }
    }
    cudaFree(dx);
    cudaFree(dg);
    cudaFree(ds);
    cudaFree(dy);
    return bad;
}

/* SkipGroupNorm on the usage example's (2, 3, 2, 8) NHWC shape, 2 groups. */
static int group_case(cudaStream_t stream) {
    enum { N = 2, H = 3, W = 2, C = 8, G = 2, NE = N * H * W * C };
    float x[NE], skip[N * C], s[NE], y[NE];
    const float gamma[C] = {1, 2, 0.5f, 1, 1, 1, -1, 3};
    const float beta[C] = {0, 0.25f, 0, -1, 0.5f, 0, 0, 0};
    const int64_t skip_dims[2] = {N, C};
    for (int n = 0; n < N; ++n)
        for (int p = 0; p < H * W; ++p)
            for (int c = 0; c < C; ++c) x[(n * H * W + p) * C + c] = (p + c) % 2 == 0 ? 1.0f : -1.0f;
    for (int c = 0; c < C; ++c) {
        skip[c] = c < 4 ? 1.0f : 2.0f;
        skip[C + c] = -0.5f;
    }
    const size_t ws_bytes = b200norm_skip_group_workspace_size(N, C, H, W, G, B200NORM_F32, 1);
    float *dx, *dskip, *dgamma, *dbeta, *dy, *ds;
    void* ws;
    int bad = 0;
    if (cudaMalloc((void**)&dx, sizeof(x)) || cudaMalloc((void**)&dskip, sizeof(skip)) ||
        cudaMalloc((void**)&dgamma, sizeof(gamma)) || cudaMalloc((void**)&dbeta, sizeof(beta)) ||
        cudaMalloc((void**)&dy, sizeof(y)) || cudaMalloc((void**)&ds, sizeof(s)) ||
        cudaMalloc(&ws, ws_bytes)) {
        fprintf(stderr, "FAIL: CUDA setup (skip_group)\n");
        return 1;
    }
    cudaMemcpy(dx, x, sizeof(x), cudaMemcpyHostToDevice);
    cudaMemcpy(dskip, skip, sizeof(skip), cudaMemcpyHostToDevice);
    cudaMemcpy(dgamma, gamma, sizeof(gamma), cudaMemcpyHostToDevice);
    cudaMemcpy(dbeta, beta, sizeof(beta), cudaMemcpyHostToDevice);
    for (int pass = 0; pass < 2; ++pass) {
        b200norm_status st;
        cudaMemset(dy, 0xFF, sizeof(y)); /* NaN patterns: every element must be written */
        cudaMemset(ds, 0xFF, sizeof(s));
        if (pass == 0) {
            st = b200norm_workspace_init(ws, ws_bytes, stream);
            if (st == B200NORM_OK)
                st = b200norm_skip_group(dx, dskip, 2, skip_dims, NULL, dgamma, dbeta, dy, ds, N,
                                         C, H, W, B200NORM_F32, B200NORM_F32, G, 0.0f, 0, 1, ws,
                                         ws_bytes, stream);
            if (st == B200NORM_OK) st = b200norm_workspace_status(ws, stream);
        } else {
            st = b200norm_skip_group_noalloc(dx, dskip, 2, skip_dims, NULL, dgamma, dbeta, dy, ds,
                                             N, C, H, W, B200NORM_F32, B200NORM_F32, G, 0.0f, 0,
                                             1, stream);
            if (st == B200NORM_OK) st = b200norm_skip_group_noalloc_status(stream);
        }
        if (st != B200NORM_OK || cudaStreamSynchronize(stream) != cudaSuccess) {
            fprintf(stderr, "FAIL: skip_group call (pass %d): %s\n", pass,
                    b200norm_last_error());
            bad = 1;
            continue;
        }
        cudaMemcpy(y, dy, sizeof(y), cudaMemcpyDeviceToHost);
        cudaMemcpy(s, ds, sizeof(s), cudaMemcpyDeviceToHost);
        for (int i = 0; i < NE; ++i) {
            const int c = i % C, n = i / (H * W * C);
            const float want_s = x[i] + skip[n * C + c];
            const double want_y = (double)gamma[c] * x[i] + beta[c];
            if (s[i] != want_s || fabs(y[i] - want_y) > 1e-6 * (1.0 + fabs(want_y))) {
                fprintf(stderr, "FAIL: skip_group (pass %d) element %d: S %.9g (want %.9g), "
                        "Y %.9g (want %.9g)\n", pass, i, s[i], want_s, y[i], want_y);
                bad = 1;
                break;
            }
        }
    }
    cudaFree(dx);
    cudaFree(dskip);
    cudaFree(dgamma);
    cudaFree(dbeta);
    cudaFree(dy);
    cudaFree(ds);
    cudaFree(ws);
    return bad;
}
#endif

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
    check(gated_case(stream) == 0, "gated_rms closed form");
    check(group_case(stream) == 0, "skip_group closed form");
    cudaStreamDestroy(stream);
#endif
    if (fails == 0) printf("ok\n");
    return fails == 0 ? 0 : 1;
}
