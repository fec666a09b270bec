/* A plain C client of libmhc (no C++, no PyTorch): allocates device buffers
 * with the CUDA runtime, fills the inputs from a fixed integer pattern, runs
 * mhc_layer_fwd and mhc_layer_bwd with workspaces sized by
 * mhc_workspace_bytes, checks every status, and writes the inputs and outputs
 * to a binary file for the test that built it.
 *
 *   layer_client T n C out.bin
 *
 * The file holds, in order: x, f, bias, dout, dy (bf16 bits), W, alpha, b
 * (fp32), then H_pre, H_post, H_res, u, r (fp32), y, out (bf16), dx, df (bf16),
 * dW, dalpha, db, dbias (fp32). */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "mhc.h"

static void die(const char *what, int code)
{
    fprintf(stderr, "layer_client: %s failed (%d): %s\n", what, code, mhc_last_error());
    exit(1);
}

#define CK(call)                                      \
    do {                                              \
        int rc_ = (int)(call);                        \
        if (rc_ != 0) die(#call, rc_);                \
    } while (0)

/* bf16 bits of a small value on a fixed grid: exact in bf16 */
static uint16_t bf16_of(float v)
{
    uint32_t u;
    memcpy(&u, &v, 4);
    return (uint16_t)(u >> 16); /* v has at most 8 significant bits: exact */
}

static float grid_value(uint64_t i, uint64_t salt)
{
    uint64_t h = (i + 1) * 0x9E3779B97F4A7C15ull ^ (salt * 0xBF58476D1CE4E5B9ull);
    h ^= h >> 31;
    return (float)((int)(h % 255) - 127) / 64.0f; /* multiples of 1/64 in [-1.98, 1.98] */
}

static void *dev_from_host(const void *h, size_t bytes)
{
    void *d = NULL;
    CK(cudaMalloc(&d, bytes > 0 ? bytes : 16));
    CK(cudaMemcpy(d, h, bytes, cudaMemcpyHostToDevice));
    return d;
}

static void *dev_alloc(size_t bytes)
{
    void *d = NULL;
    CK(cudaMalloc(&d, bytes > 0 ? bytes : 16));
    return d;
}

static void dump(FILE *fp, const void *d, size_t bytes)
{
    void *h = malloc(bytes > 0 ? bytes : 1);
    CK(cudaMemcpy(h, d, bytes, cudaMemcpyDeviceToHost));
    if (fwrite(h, 1, bytes, fp) != bytes) die("fwrite", -1);
    free(h);
}

int main(int argc, char **argv)
{
    if (argc != 5) {
        fprintf(stderr, "usage: layer_client T n C out.bin\n");
        return 2;
    }
    const int64_t T = atoll(argv[1]), C = atoll(argv[3]);
    const int n = atoi(argv[2]);
    const int64_t K = n * C, O = (int64_t)n * n + 2 * n;
    const int iters = 20;
    const float eps = 1e-6f;

    uint16_t *x = malloc(T * K * 2), *f = malloc(T * C * 2), *bias = malloc(C * 2);
    uint16_t *dout = malloc(T * K * 2), *dy = malloc(T * C * 2);
    float *W = malloc(K * O * 4), alpha[3] = {0.01f, 0.01f, 0.01f}, *b = malloc(O * 4);
    for (int64_t i = 0; i < T * K; ++i) x[i] = bf16_of(grid_value(i, 1));
    for (int64_t i = 0; i < T * C; ++i) f[i] = bf16_of(grid_value(i, 2));
    for (int64_t i = 0; i < C; ++i) bias[i] = bf16_of(grid_value(i, 3) / 64.0f);
    for (int64_t i = 0; i < T * K; ++i) dout[i] = bf16_of(grid_value(i, 4));
    for (int64_t i = 0; i < T * C; ++i) dy[i] = bf16_of(grid_value(i, 5));
    for (int64_t i = 0; i < K * O; ++i) W[i] = grid_value(i, 6) / 64.0f;
    for (int64_t i = 0; i < O; ++i) b[i] = grid_value(i, 7) / 4.0f;

    void *dx_in = dev_from_host(x, T * K * 2), *df_in = dev_from_host(f, T * C * 2);
    void *dbias_in = dev_from_host(bias, C * 2), *ddout = dev_from_host(dout, T * K * 2);
    void *ddy = dev_from_host(dy, T * C * 2), *dW_in = dev_from_host(W, K * O * 4);
    void *dalpha_in = dev_from_host(alpha, 12), *db_in = dev_from_host(b, O * 4);

    float *Hpre = dev_alloc(T * n * 4), *Hpost = dev_alloc(T * n * 4);
    float *Hres = dev_alloc(T * n * n * 4), *u = dev_alloc(T * O * 4), *r = dev_alloc(T * 4);
    mhc_bf16 *y = dev_alloc(T * C * 2), *out = dev_alloc(T * K * 2);
    mhc_bf16 *gx = dev_alloc(T * K * 2), *gf = dev_alloc(T * C * 2);
    float *gW = dev_alloc(K * O * 4), *galpha = dev_alloc(12), *gb = dev_alloc(O * 4);
    float *gbias = dev_alloc(C * 4);

    const size_t wsf_b = mhc_workspace_bytes(MHC_OP_LAYER_FWD, T, n, C);
    const size_t wsb_b = mhc_workspace_bytes(MHC_OP_LAYER_BWD, T, n, C);
    if (wsf_b == 0 || wsb_b == 0) die("mhc_workspace_bytes", 0);
    void *wsf = dev_alloc(wsf_b), *wsb = dev_alloc(wsb_b);

    CK(mhc_layer_fwd(dx_in, dW_in, dalpha_in, db_in, df_in, dbias_in, T, n, C, iters, eps, eps,
                     Hpre, Hpost, Hres, u, r, y, out, wsf, wsf_b, NULL));
    CK(mhc_layer_bwd(ddout, ddy, dx_in, dW_in, dalpha_in, db_in, df_in, dbias_in, Hpre, Hpost,
                     Hres, u, r, T, n, C, iters, eps, eps, gx, gf, gW, galpha, gb, gbias, wsb,
                     wsb_b, NULL));
    /* a too-small workspace is refused before any launch */
    if (mhc_layer_bwd(ddout, ddy, dx_in, dW_in, dalpha_in, db_in, df_in, dbias_in, Hpre, Hpost,
                      Hres, u, r, T, n, C, iters, eps, eps, gx, gf, gW, galpha, gb, gbias, wsb,
                      wsb_b - 256, NULL) != MHC_ERR_WORKSPACE_TOO_SMALL)
        die("workspace check", -2);
    CK(cudaDeviceSynchronize());
    int code = 0;
    CK(mhc_device_error(&code, NULL));

    FILE *fp = fopen(argv[4], "wb");
    if (!fp) die("fopen", -1);
    fwrite(x, 2, T * K, fp);
    fwrite(f, 2, T * C, fp);
    fwrite(bias, 2, C, fp);
    fwrite(dout, 2, T * K, fp);
    fwrite(dy, 2, T * C, fp);
    fwrite(W, 4, K * O, fp);
    fwrite(alpha, 4, 3, fp);
    fwrite(b, 4, O, fp);
    dump(fp, Hpre, T * n * 4);
    dump(fp, Hpost, T * n * 4);
    dump(fp, Hres, T * n * n * 4);
    dump(fp, u, T * O * 4);
    dump(fp, r, T * 4);
    dump(fp, y, T * C * 2);
    dump(fp, out, T * K * 2);
    dump(fp, gx, T * K * 2);
    dump(fp, gf, T * C * 2);
    dump(fp, gW, K * O * 4);
    dump(fp, galpha, 12);
    dump(fp, gb, O * 4);
    dump(fp, gbias, C * 4);
    fclose(fp);
    printf("layer_client ok: T=%lld n=%d C=%lld\n", (long long)T, n, (long long)C);
    return 0;
}
