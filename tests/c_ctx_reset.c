/* c_ctx_reset.c -- a C11 caller that runs the library's fast paths, destroys
 * its CUDA context with cudaDeviceReset, and runs them again in the new
 * context: every call must succeed there too and give the same bytes.  The
 * library caches per device what belongs to a context (the kernels' shared
 * memory limits, its workspace pool, the address of the fixed scratch
 * array), so a call after the reset must notice the new context.  Needs a GPU;
 * prints "ctx reset check: ok" and exits 0 on success. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "ssmscan.h"

static int fails = 0;

#define CHECK_CUDA(x)                                                          \
    do {                                                                       \
        cudaError_t e_ = (x);                                                  \
        if (e_ != cudaSuccess) {                                               \
            printf("FAIL %s: %s\n", #x, cudaGetErrorString(e_));               \
            exit(1);                                                           \
        }                                                                      \
    } while (0)

static void expect_ok(int st, const char *what) {
    if (st != SSM_OK) {
        printf("FAIL %s: %s\n", what, ssm_status_string(st));
        ++fails;
    }
}

/* deterministic values in about [-1, 1] */
static float val(uint32_t i, uint32_t salt) {
    uint32_t x = i * 2654435761u ^ (salt * 40503u + 0x9E3779B9u);
    x ^= x >> 15;
    x *= 2246822519u;
    x ^= x >> 13;
    return (float)(x & 0xFFFF) / 32768.0f - 1.0f;
}

static uint16_t to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);   /* round to nearest even */
    return (uint16_t)(u >> 16);
}

/* a device copy of n values: float32 (bf == 0) or bf16 */
static void *dev_vals(size_t n, uint32_t salt, float scale, float shift, int bf) {
    size_t i, es = bf ? 2 : 4;
    unsigned char *h = (unsigned char *)malloc(n * es);
    void *d = NULL;
    for (i = 0; i < n; ++i) {
        float v = val((uint32_t)i, salt) * scale + shift;
        if (bf) {
            uint16_t b = to_bf16(v);
            memcpy(h + 2 * i, &b, 2);
        } else {
            memcpy(h + 4 * i, &v, 4);
        }
    }
    CHECK_CUDA(cudaMalloc(&d, n * es));
    CHECK_CUDA(cudaMemcpy(d, h, n * es, cudaMemcpyHostToDevice));
    free(h);
    return d;
}

static void *dev_zero(size_t bytes) {
    void *d = NULL;
    CHECK_CUDA(cudaMalloc(&d, bytes));
    CHECK_CUDA(cudaMemset(d, 0, bytes));
    return d;
}

static unsigned char *to_host(const void *d, size_t bytes) {
    unsigned char *h = (unsigned char *)malloc(bytes);
    CHECK_CUDA(cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost));
    return h;
}

/* A-matrix -(n+1) per channel */
static float *dev_A(int64_t D, int64_t N) {
    int64_t d, n;
    float *h = (float *)malloc((size_t)(D * N) * 4);
    void *p = NULL;
    for (d = 0; d < D; ++d)
        for (n = 0; n < N; ++n) h[d * N + n] = -(float)(n + 1);
    CHECK_CUDA(cudaMalloc(&p, (size_t)(D * N) * 4));
    CHECK_CUDA(cudaMemcpy(p, h, (size_t)(D * N) * 4, cudaMemcpyHostToDevice));
    free(h);
    return (float *)p;
}

enum { NOUT = 6 };

/* Runs the fast paths once on fresh device buffers; returns host copies of
 * their outputs in out[], sizes in len[]. */
static void run_all(unsigned char *out[NOUT], size_t len[NOUT]) {
    /* scan (bf16, N = 16, the chained plan with a workspace) */
    const int64_t b = 2, L = 512, D = 512, N = 16;
    const size_t nx = (size_t)(b * L * D), nbc = (size_t)(b * L * N);
    void *u = dev_vals(nx, 1, 1.0f, 0.0f, 1), *dl = dev_vals(nx, 2, 1.0f, 0.0f, 1);
    void *z = dev_vals(nx, 3, 1.0f, 0.0f, 1), *B = dev_vals(nbc, 4, 1.0f, 0.0f, 1);
    void *C = dev_vals(nbc, 5, 1.0f, 0.0f, 1);
    float *bias = (float *)dev_vals((size_t)D, 6, 1.0f, -4.0f, 0);
    float *dsk = (float *)dev_vals((size_t)D, 7, 1.0f, 0.0f, 0);
    float *A = dev_A(D, N);
    void *y = dev_zero(nx * 2), *y2 = dev_zero(nx * 2);
    float *h = (float *)dev_zero((size_t)(b * D * N) * 4);
    /* decode (bf16, the tiled kernel) */
    const int64_t sb = 8;
    void *su = dev_vals((size_t)(sb * D), 11, 1.0f, 0.0f, 1);
    void *sd = dev_vals((size_t)(sb * D), 12, 1.0f, 0.0f, 1);
    void *sz = dev_vals((size_t)(sb * D), 13, 1.0f, 0.0f, 1);
    void *sB = dev_vals((size_t)(sb * N), 14, 1.0f, 0.0f, 1);
    void *sC = dev_vals((size_t)(sb * N), 15, 1.0f, 0.0f, 1);
    float *state = (float *)dev_vals((size_t)(sb * D * N), 16, 1.0f, 0.0f, 0);
    void *sy = dev_zero((size_t)(sb * D) * 2);
    /* SSD (bf16, P = 64, N = 64, the tensor-core kernel) */
    const int64_t H = 2, P = 64, NS = 64, LS = 256;
    void *x = dev_vals((size_t)(LS * H * P), 21, 1.0f, 0.0f, 1);
    void *dt = dev_vals((size_t)(LS * H), 22, 1.0f, 0.0f, 1);
    void *SB = dev_vals((size_t)(LS * NS), 23, 1.0f, 0.0f, 1);
    void *SC = dev_vals((size_t)(LS * NS), 24, 1.0f, 0.0f, 1);
    float *Ah = (float *)dev_vals((size_t)H, 25, 0.5f, -1.0f, 0);
    float *bh = (float *)dev_vals((size_t)H, 26, 1.0f, -3.0f, 0);
    void *xy = dev_zero((size_t)(LS * H * P) * 2);
    float *hs = (float *)dev_zero((size_t)(H * P * NS) * 4);
    /* backward (bf16) */
    void *dy = dev_vals(nx, 31, 1.0f, 0.0f, 1);
    void *du = dev_zero(nx * 2), *ddl = dev_zero(nx * 2), *dz = dev_zero(nx * 2);
    float *ddb = (float *)dev_zero((size_t)D * 4), *dA = (float *)dev_zero((size_t)(D * N) * 4);
    float *dB = (float *)dev_zero(nbc * 4), *dC = (float *)dev_zero(nbc * 4);
    float *dD = (float *)dev_zero((size_t)D * 4);

    expect_ok(ssm_scan_fwd(u, dl, bias, A, B, C, dsk, z, y, h, b, L, D, N, SSM_BF16, NULL),
              "ssm_scan_fwd");
    expect_ok(ssm_scan_fwd_noalloc(u, dl, bias, A, B, C, dsk, z, y2, NULL, b, L, D, N, SSM_BF16,
                                   NULL),
              "ssm_scan_fwd_noalloc");
    expect_ok(ssm_step(state, su, sd, bias, A, sB, sC, dsk, sz, sy, sb, D, N, SSM_BF16, NULL),
              "ssm_step");
    expect_ok(ssm_ssd_fwd(x, dt, bh, Ah, SB, SC, NULL, xy, hs, 1, LS, H, P, NS, SSM_BF16, NULL),
              "ssm_ssd_fwd");
    expect_ok(ssm_scan_bwd(u, dl, bias, A, B, C, dsk, z, dy, NULL, du, ddl, ddb, dA, dB, dC, dD,
                           dz, b, L, D, N, SSM_BF16, NULL),
              "ssm_scan_bwd");
    CHECK_CUDA(cudaDeviceSynchronize());
    expect_ok(ssm_device_status(NULL), "device status");

    out[0] = to_host(y, nx * 2);
    len[0] = nx * 2;
    out[1] = to_host(y2, nx * 2);
    len[1] = nx * 2;
    out[2] = to_host(sy, (size_t)(sb * D) * 2);
    len[2] = (size_t)(sb * D) * 2;
    out[3] = to_host(xy, (size_t)(LS * H * P) * 2);
    len[3] = (size_t)(LS * H * P) * 2;
    out[4] = to_host(du, nx * 2);
    len[4] = nx * 2;
    out[5] = to_host(h, (size_t)(b * D * N) * 4);
    len[5] = (size_t)(b * D * N) * 4;
    /* the buffers go with the context */
}

int main(void) {
    unsigned char *first[NOUT], *second[NOUT];
    size_t len1[NOUT], len2[NOUT];
    int i;
    const char *names[NOUT] = {"scan y", "noalloc y", "step y", "ssd y", "bwd du", "scan h_last"};
    CHECK_CUDA(cudaSetDevice(0));
    run_all(first, len1);
    CHECK_CUDA(cudaDeviceReset());
    run_all(second, len2);
    for (i = 0; i < NOUT; ++i) {
        if (len1[i] != len2[i] || memcmp(first[i], second[i], len1[i]) != 0) {
            printf("FAIL %s differs after the reset\n", names[i]);
            ++fails;
        }
        free(first[i]);
        free(second[i]);
    }
    CHECK_CUDA(cudaDeviceReset());
    if (fails) {
        printf("ctx reset check: %d failures\n", fails);
        return 1;
    }
    printf("ctx reset check: ok\n");
    return 0;
}
