// Bit-reproducible mode: the mHC ops with the pinned reduction trees of the
// RL-Align/RL-Kernel PR #383 numerical contract (PR body, "Numerical
// contract": only a serial ascending left fold for long reductions and
// (a0 + a1) + (a2 + a3) over the four streams; fp32 arithmetic).  n = 4.
//
//   fold4(a0..a3) = (a0 + a1) + (a2 + a3)
//   fold(v)       = ((0 + v_0) + v_1) + ... in ascending index order
//
// Every operation is an explicitly rounded intrinsic (__fadd_rn, __fmul_rn,
// __fdiv_rn, __fsqrt_rn; __fmaf_rn only inside exp), so the compiler
// contracts nothing and the results are the same bits on any device and
// any run, and the same bits as a plain fp32 program that performs the same
// operations in the same order.  exp is the mode's own (pin_exp): Cody and
// Waite's reduction x = n ln2 + r, the Taylor series of e^r to degree 7 in
// Horner form, exact scaling by 2^n; CUDA's expf is not used because its
// last bit is not specified.  The operation order of each formula is the
// left-to-right reading written next to it.
//
// The kernels are plain thread-per-output loops: the mode exists to make
// results reproducible across devices and implementations, not to be fast
// (the sums over channels and tokens are serial by contract).
#include <atomic>

#include "launch.h"

namespace mhc {

namespace {

constexpr int PN = 4, PO = PN * PN + 2 * PN;

__device__ __forceinline__ float add(float a, float b) { return __fadd_rn(a, b); }
__device__ __forceinline__ float sub(float a, float b) { return __fsub_rn(a, b); }
__device__ __forceinline__ float mul(float a, float b) { return __fmul_rn(a, b); }
__device__ __forceinline__ float dvd(float a, float b) { return __fdiv_rn(a, b); }
__device__ __forceinline__ float fold4(float a0, float a1, float a2, float a3)
{
    return add(add(a0, a1), add(a2, a3));
}
__device__ __forceinline__ float bf(bf16 v) { return __bfloat162float(v); }

__device__ float pin_exp(float x)
{
    x = fminf(fmaxf(x, -87.0f), 88.0f);   // keeps the result a normal fp32 value
    const float log2e = 0x1.715476p+0f;
    const float ln2_hi = 0x1.62e4p-1f;     // 12 significant bits: n * ln2_hi is exact
    const float ln2_lo = 0x1.7f7d1cp-20f;  // ln2 - ln2_hi
    const float n = rintf(mul(x, log2e));
    float r = __fmaf_rn(-n, ln2_hi, x);
    r = __fmaf_rn(-n, ln2_lo, r);
    float p = 0x1.a01a02p-13f;             // 1/7!, then 1/6!, ..., 1/3!
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);
    p = __fmaf_rn(p, r, 0x1.111112p-7f);
    p = __fmaf_rn(p, r, 0x1.555556p-5f);
    p = __fmaf_rn(p, r, 0x1.555556p-3f);
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    return mul(p, __int_as_float((int(n) + 127) << 23));
}

__device__ __forceinline__ float pin_sigmoid(float z) { return dvd(1.0f, add(1.0f, pin_exp(-z))); }

// Sinkhorn of one 4 x 4 matrix (row step then column step, `iters` times,
// each line divided by (its fold4 sum + eps)); trace[2k] after the row step
// of iteration k, trace[2k+1] after its column step.
__device__ void pin_sinkhorn(const float *z, int iters, float eps, float *A, float *trace)
{
    for (int e = 0; e < PN * PN; ++e) A[e] = pin_exp(z[e]);
    for (int k = 0; k < iters; ++k) {
        for (int i = 0; i < PN; ++i) {
            const float d = add(fold4(A[i * PN], A[i * PN + 1], A[i * PN + 2], A[i * PN + 3]), eps);
            for (int j = 0; j < PN; ++j) A[i * PN + j] = dvd(A[i * PN + j], d);
        }
        if (trace)
            for (int e = 0; e < PN * PN; ++e) trace[(2 * k) * PN * PN + e] = A[e];
        for (int j = 0; j < PN; ++j) {
            const float d = add(fold4(A[j], A[PN + j], A[2 * PN + j], A[3 * PN + j]), eps);
            for (int i = 0; i < PN; ++i) A[i * PN + j] = dvd(A[i * PN + j], d);
        }
        if (trace)
            for (int e = 0; e < PN * PN; ++e) trace[(2 * k + 1) * PN * PN + e] = A[e];
    }
}

// Gradient of pin_sinkhorn: per step X -> Y = X / d, dX = (dY - fold4(dY Y)) / d,
// columns then rows from the last iteration back; dz = G exp(z).
__device__ void pin_sinkhorn_bwd(const float *g_in, const float *z, int iters, float eps, float *dz,
                                 float *trace)
{
    float P[PN * PN], E[PN * PN], G[PN * PN];
    pin_sinkhorn(z, iters, eps, P, trace);
    for (int e = 0; e < PN * PN; ++e) {
        E[e] = pin_exp(z[e]);
        G[e] = g_in[e];
    }
    for (int k = iters - 1; k >= 0; --k) {
        const float *Bk = trace + (2 * k) * PN * PN;
        const float *Ak = trace + (2 * k + 1) * PN * PN;
        const float *Ap = (k == 0) ? E : trace + (2 * k - 1) * PN * PN;
        for (int j = 0; j < PN; ++j) {
            const float d = add(fold4(Bk[j], Bk[PN + j], Bk[2 * PN + j], Bk[3 * PN + j]), eps);
            const float dot = fold4(mul(G[j], Ak[j]), mul(G[PN + j], Ak[PN + j]),
                                    mul(G[2 * PN + j], Ak[2 * PN + j]), mul(G[3 * PN + j], Ak[3 * PN + j]));
            for (int i = 0; i < PN; ++i) G[i * PN + j] = dvd(sub(G[i * PN + j], dot), d);
        }
        for (int i = 0; i < PN; ++i) {
            const float *a = Ap + i * PN, *bb = Bk + i * PN;
            float *gg = G + i * PN;
            const float d = add(fold4(a[0], a[1], a[2], a[3]), eps);
            const float dot = fold4(mul(gg[0], bb[0]), mul(gg[1], bb[1]), mul(gg[2], bb[2]),
                                    mul(gg[3], bb[3]));
            for (int j = 0; j < PN; ++j) gg[j] = dvd(sub(gg[j], dot), d);
        }
    }
    for (int e = 0; e < PN * PN; ++e) dz[e] = mul(G[e], E[e]);
}

__device__ __forceinline__ float seg_alpha(const float *alpha, int o)
{
    return o < PN ? alpha[0] : (o < 2 * PN ? alpha[1] : alpha[2]);
}

// one token: s = fold_k x^2, u[o] = fold_k x[k] W[k][o], q = sqrt(s / K), r = 1 / (q + eps)
__device__ void pin_proj_token(const bf16 *xt, const float *W, int64_t K, float eps_rms, float *u,
                               float &q, float &r)
{
    float s = 0.0f;
    for (int o = 0; o < PO; ++o) u[o] = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
        const float xv = bf(xt[k]);
        s = add(s, mul(xv, xv));
        const float *wk = W + k * PO;
#pragma unroll
        for (int o = 0; o < PO; ++o) u[o] = add(u[o], mul(xv, __ldg(wk + o)));
    }
    q = __fsqrt_rn(dvd(s, float(K)));
    r = dvd(1.0f, add(q, eps_rms));
}

// z[o] = (alpha_seg r) u[o] + b[o]
__device__ __forceinline__ float pin_logit(const float *u, float r, const float *alpha,
                                           const float *b, int o)
{
    return add(mul(mul(seg_alpha(alpha, o), r), u[o]), b[o]);
}

// ---------------------------------------------------------------------------
// kernels
// ---------------------------------------------------------------------------

__global__ void k_pin_sinkhorn_fwd(const float *__restrict__ lg, float *__restrict__ P, int64_t M,
                                   int iters, float eps)
{
    pdl_wait();
    const int64_t m = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (m >= M) return;
    float A[PN * PN];
    pin_sinkhorn(lg + m * PN * PN, iters, eps, A, nullptr);
    for (int e = 0; e < PN * PN; ++e) P[m * PN * PN + e] = A[e];
}

// the forward's intermediate matrices live in the thread's local memory
__global__ void k_pin_sinkhorn_bwd(const float *__restrict__ dP, const float *__restrict__ lg,
                                   float *__restrict__ dl, int64_t M, int iters, float eps)
{
    pdl_wait();
    const int64_t m = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (m >= M) return;
    float trace[2 * kMaxIters * PN * PN];
    pin_sinkhorn_bwd(dP + m * PN * PN, lg + m * PN * PN, iters, eps, dl + m * PN * PN, trace);
}

// proj_rms_compute_h forward, a thread per token
__global__ void k_pin_proj_fwd(const bf16 *__restrict__ x, const float *__restrict__ W,
                               const float *__restrict__ alpha, const float *__restrict__ b,
                               int64_t T, int64_t C, int iters, float eps_sk, float eps_rms,
                               float *Hpre, float *Hpost, float *Hres, float *u_save,
                               float *r_save)
{
    pdl_wait();
    const int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= T) return;
    const int64_t K = PN * C;
    float u[PO], z[PO], q, r, A[PN * PN];
    pin_proj_token(x + t * K, W, K, eps_rms, u, q, r);
    for (int o = 0; o < PO; ++o) z[o] = pin_logit(u, r, alpha, b, o);
    for (int i = 0; i < PN; ++i) {
        Hpre[t * PN + i] = pin_sigmoid(z[i]);
        Hpost[t * PN + i] = mul(2.0f, pin_sigmoid(z[PN + i]));
    }
    pin_sinkhorn(z + 2 * PN, iters, eps_sk, A, nullptr);
    for (int e = 0; e < PN * PN; ++e) Hres[t * PN * PN + e] = A[e];
    if (u_save)
        for (int o = 0; o < PO; ++o) u_save[t * PO + o] = u[o];
    if (r_save) r_save[t] = r;
}

// Per-token backward quantities, a thread per token (u, q, r recomputed from x):
//   dz_pre = (dH_pre s) (1 - s), dz_post = ((2 dH_post) s) (1 - s), dz_res = Sinkhorn bwd,
//   g_seg = fold_{o in seg} dz u, ga_seg = g_seg r, dr = fold_seg alpha_seg g_seg,
//   du = (alpha_seg r) dz, coef = ((-dr r) r) / (K q) (0 when q = 0).
// Out: du, dz [T][PO], ga [T][3], coef [T].
__global__ void k_pin_bwd_token(const float *__restrict__ dHpre, const float *__restrict__ dHpost,
                                const float *__restrict__ dHres, const bf16 *__restrict__ x,
                                const float *__restrict__ W, const float *__restrict__ alpha,
                                const float *__restrict__ b, int64_t T, int64_t C, int iters,
                                float eps_sk, float eps_rms, float *__restrict__ du,
                                float *__restrict__ dz_out, float *__restrict__ ga,
                                float *__restrict__ coef)
{
    pdl_wait();
    const int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (t >= T) return;
    const int64_t K = PN * C;
    float u[PO], z[PO], dz[PO], q, r;
    float trace[2 * kMaxIters * PN * PN];   // the Sinkhorn forward's steps, local memory
    pin_proj_token(x + t * K, W, K, eps_rms, u, q, r);
    for (int o = 0; o < PO; ++o) z[o] = pin_logit(u, r, alpha, b, o);
    for (int i = 0; i < PN; ++i) {
        const float sp = pin_sigmoid(z[i]), so = pin_sigmoid(z[PN + i]);
        dz[i] = mul(mul(dHpre[t * PN + i], sp), sub(1.0f, sp));
        dz[PN + i] = mul(mul(mul(2.0f, dHpost[t * PN + i]), so), sub(1.0f, so));
    }
    pin_sinkhorn_bwd(dHres + t * PN * PN, z + 2 * PN, iters, eps_sk, dz + 2 * PN, trace);
    float g[3] = {0.0f, 0.0f, 0.0f};
    for (int o = 0; o < PO; ++o) {
        const int sg = o < PN ? 0 : (o < 2 * PN ? 1 : 2);
        g[sg] = add(g[sg], mul(dz[o], u[o]));
    }
    float dr = 0.0f;
    for (int s = 0; s < 3; ++s) {
        ga[t * 3 + s] = mul(g[s], r);
        dr = add(dr, mul(alpha[s], g[s]));
    }
    for (int o = 0; o < PO; ++o) {
        du[t * PO + o] = mul(mul(seg_alpha(alpha, o), r), dz[o]);
        dz_out[t * PO + o] = dz[o];
    }
    coef[t] = (q > 0.0f) ? dvd(mul(mul(-dr, r), r), mul(float(K), q)) : 0.0f;
}

// dx, a thread per element (t, k = j C + c):
//   dx_proj = fold_o(du[o] W[k][o]) + coef x[k]
//   standalone: dx = bf16(dx_proj); layer: dx = bf16((fold4_i(H_res[j][i] dout[i][c])
//   + H_pre[j] dy[c]) + dx_proj)
__global__ void k_pin_dx(const bf16 *__restrict__ x, const float *__restrict__ W,
                         const float *__restrict__ du, const float *__restrict__ coef, int64_t T,
                         int64_t C, const bf16 *__restrict__ dout, const bf16 *__restrict__ dy,
                         const float *__restrict__ Hpre, const float *__restrict__ Hres,
                         bf16 *__restrict__ dx)
{
    pdl_wait();
    const int64_t K = PN * C;
    const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= T * K) return;
    const int64_t t = e / K, k = e % K;
    const int j = int(k / C);
    const int64_t c = k % C;
    float acc = 0.0f;
    const float *wk = W + k * PO, *dut = du + t * PO;
#pragma unroll
    for (int o = 0; o < PO; ++o) acc = add(acc, mul(dut[o], __ldg(wk + o)));
    float v = add(acc, mul(coef[t], bf(x[e])));
    if (dout) {
        const float *hr = Hres + t * PN * PN + j * PN;
        const bf16 *dt = dout + t * K + c;
        const float dres = fold4(mul(hr[0], bf(dt[0])), mul(hr[1], bf(dt[C])),
                                 mul(hr[2], bf(dt[2 * C])), mul(hr[3], bf(dt[3 * C])));
        const float dagg = mul(Hpre[t * PN + j], bf(dy[t * C + c]));
        v = add(add(dres, dagg), v);
    }
    dx[e] = __float2bfloat16_rn(v);
}

// dW[k][o] = fold_t x[t][k] du[t][o], a thread per (k, o)
__global__ void k_pin_dw(const bf16 *__restrict__ x, const float *__restrict__ du, int64_t T,
                         int64_t K, float *__restrict__ dW)
{
    pdl_wait();
    const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= K * PO) return;
    const int64_t k = e / PO;
    const int o = int(e % PO);
    float acc = 0.0f;
    for (int64_t t = 0; t < T; ++t) acc = add(acc, mul(bf(x[t * K + k]), du[t * PO + o]));
    dW[e] = acc;
}

// Column folds over tokens: out[col] = fold_t src[t][col] for col < cols
// (db from dz [T][PO]; dalpha from ga [T][3]).
__global__ void k_pin_colfold(const float *__restrict__ src, int64_t T, int cols,
                              float *__restrict__ out)
{
    pdl_wait();
    const int col = int(blockIdx.x) * blockDim.x + threadIdx.x;
    if (col >= cols) return;
    float acc = 0.0f;
    for (int64_t t = 0; t < T; ++t) acc = add(acc, src[t * cols + col]);
    out[col] = acc;
}

// y[t][c] = bf16(fold4(H_pre[i] x[i][c])), a thread per (t, c)
__global__ void k_pin_agg_fwd(const bf16 *__restrict__ x, const float *__restrict__ Hpre, int64_t T,
                              int64_t C, bf16 *__restrict__ y)
{
    pdl_wait();
    const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= T * C) return;
    const int64_t t = e / C, c = e % C;
    const bf16 *xt = x + t * PN * C + c;
    const float *h = Hpre + t * PN;
    y[e] = __float2bfloat16_rn(fold4(mul(h[0], bf(xt[0])), mul(h[1], bf(xt[C])),
                                     mul(h[2], bf(xt[2 * C])), mul(h[3], bf(xt[3 * C]))));
}

// dx[t][i][c] = bf16(H_pre[t][i] dy[t][c]), a thread per element
__global__ void k_pin_agg_bwd_dx(const bf16 *__restrict__ dy, const float *__restrict__ Hpre,
                                 int64_t T, int64_t C, bf16 *__restrict__ dx)
{
    pdl_wait();
    const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= T * PN * C) return;
    const int64_t t = e / (PN * C), c = e % C;
    const int i = int((e / C) % PN);
    dx[e] = __float2bfloat16_rn(mul(Hpre[t * PN + i], bf(dy[t * C + c])));
}

// Per-token channel folds, a thread per (t, slot):
//   slots [0,16):  dH_res[j][i] = fold_c x[j][c] dout[i][c]       (dout given)
//   slots [16,20): dH_post[i]   = fold_c dout[i][c] (f[c] + bias[c]) (dout given)
//   slots [20,24): dH_pre[i]    = fold_c dy[c] x[i][c]            (dy given)
__global__ void k_pin_tok_folds(const bf16 *__restrict__ x, const bf16 *__restrict__ dout,
                                const bf16 *__restrict__ f, const bf16 *__restrict__ bias,
                                const bf16 *__restrict__ dy, int64_t T, int64_t C,
                                float *__restrict__ dHres, float *__restrict__ dHpost,
                                float *__restrict__ dHpre)
{
    pdl_wait();
    const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= T * 24) return;
    const int64_t t = e / 24;
    const int slot = int(e % 24);
    const bf16 *xt = x + t * PN * C;
    float acc = 0.0f;
    if (slot < 16) {
        if (!dout) return;
        const int j = slot / PN, i = slot % PN;
        const bf16 *a = xt + j * C, *g = dout + t * PN * C + i * C;
        for (int64_t c = 0; c < C; ++c) acc = add(acc, mul(bf(a[c]), bf(g[c])));
        dHres[t * PN * PN + slot] = acc;
    } else if (slot < 20) {
        if (!dout) return;
        const int i = slot - 16;
        const bf16 *g = dout + t * PN * C + i * C, *ft = f + t * C;
        for (int64_t c = 0; c < C; ++c)
            acc = add(acc, mul(bf(g[c]), add(bf(ft[c]), bias ? bf(bias[c]) : 0.0f)));
        dHpost[t * PN + i] = acc;
    } else {
        if (!dy) return;
        const int i = slot - 20;
        const bf16 *a = xt + i * C, *d = dy + t * C;
        for (int64_t c = 0; c < C; ++c) acc = add(acc, mul(bf(d[c]), bf(a[c])));
        dHpre[t * PN + i] = acc;
    }
}

// out[t][i][c] = bf16(fold4_j(H_res[j][i] x[j][c]) + H_post[i] (f[c] + bias[c])), a thread per (t, c)
__global__ void k_pin_post_fwd(const bf16 *__restrict__ res, const bf16 *__restrict__ f,
                               const bf16 *__restrict__ bias, const float *__restrict__ Hres,
                               const float *__restrict__ Hpost, int64_t T, int64_t C,
                               bf16 *__restrict__ out)
{
    pdl_wait();
    const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= T * C) return;
    const int64_t t = e / C, c = e % C;
    const float g = add(bf(f[e]), bias ? bf(bias[c]) : 0.0f);
    const bf16 *xr = res + t * PN * C + c;
    const float *hr = Hres + t * PN * PN;
    const float x0 = bf(xr[0]), x1 = bf(xr[C]), x2 = bf(xr[2 * C]), x3 = bf(xr[3 * C]);
    for (int i = 0; i < PN; ++i) {
        const float m = fold4(mul(hr[i], x0), mul(hr[PN + i], x1), mul(hr[2 * PN + i], x2),
                              mul(hr[3 * PN + i], x3));
        out[(t * PN + i) * C + c] = __float2bfloat16_rn(add(m, mul(Hpost[t * PN + i], g)));
    }
}

// post_bda backward elementwise part, a thread per (t, c):
//   dfv = fold4_i(H_post[i] dout[i][c]) -> df = bf16(dfv);
//   dres[j][c] = bf16(fold4_i(H_res[j][i] dout[i][c]))
__global__ void k_pin_post_bwd_elem(const bf16 *__restrict__ dout, const float *__restrict__ Hres,
                                    const float *__restrict__ Hpost, int64_t T, int64_t C,
                                    bf16 *__restrict__ dres, bf16 *__restrict__ df)
{
    pdl_wait();
    const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= T * C) return;
    const int64_t t = e / C, c = e % C;
    const bf16 *dt = dout + t * PN * C + c;
    const float d0 = bf(dt[0]), d1 = bf(dt[C]), d2 = bf(dt[2 * C]), d3 = bf(dt[3 * C]);
    const float *hp = Hpost + t * PN, *hr = Hres + t * PN * PN;
    if (df) df[e] = __float2bfloat16_rn(fold4(mul(hp[0], d0), mul(hp[1], d1), mul(hp[2], d2), mul(hp[3], d3)));
    if (dres)
        for (int j = 0; j < PN; ++j)
            dres[(t * PN + j) * C + c] = __float2bfloat16_rn(
                fold4(mul(hr[j * PN], d0), mul(hr[j * PN + 1], d1), mul(hr[j * PN + 2], d2),
                      mul(hr[j * PN + 3], d3)));
}

// dbias[c] = fold_t fold4_i(H_post[t][i] dout[t][i][c]), a thread per channel
__global__ void k_pin_dbias(const bf16 *__restrict__ dout, const float *__restrict__ Hpost,
                            int64_t T, int64_t C, float *__restrict__ dbias)
{
    pdl_wait();
    const int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (c >= C) return;
    float acc = 0.0f;
    for (int64_t t = 0; t < T; ++t) {
        const bf16 *dt = dout + t * PN * C + c;
        const float *hp = Hpost + t * PN;
        acc = add(acc, fold4(mul(hp[0], bf(dt[0])), mul(hp[1], bf(dt[C])), mul(hp[2], bf(dt[2 * C])),
                             mul(hp[3], bf(dt[3 * C]))));
    }
    dbias[c] = acc;
}

unsigned blocks(int64_t n, int per = 128) { return unsigned((n + per - 1) / per); }

}  // namespace

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static std::atomic<int> g_pinned{0};
void set_pinned(int on) { g_pinned.store(on ? 1 : 0, std::memory_order_relaxed); }
int pinned() { return g_pinned.load(std::memory_order_relaxed); }

// backward scratch: du, dz [T][PO], ga [T][3], coef [T], dH_pre, dH_post [T][4],
// dH_res [T][16]
size_t pin_bwd_ws_bytes(int64_t T) { return ws_align(size_t(T) * (2 * PO + 3 + 1 + PN + PN + PN * PN) * 4); }

cudaError_t launch_pin_sinkhorn_fwd(const float *lg, float *P, int64_t M, int iters, float eps,
                                    cudaStream_t s)
{
    MHC_PROF("k_pin_sinkhorn_fwd", s);
    launch_k(k_pin_sinkhorn_fwd, dim3(blocks(M)), dim3(128), 0, s, lg, P, M, iters, eps);
    return cudaGetLastError();
}

cudaError_t launch_pin_sinkhorn_bwd(const float *dP, const float *lg, float *dl, int64_t M,
                                    int iters, float eps, cudaStream_t s)
{
    MHC_PROF("k_pin_sinkhorn_bwd", s);
    launch_k(k_pin_sinkhorn_bwd, dim3(blocks(M, 64)), dim3(64), 0, s, dP, lg, dl, M, iters, eps);
    return cudaGetLastError();
}

cudaError_t launch_pin_proj_fwd(const bf16 *x, const float *W, const float *alpha, const float *b,
                                int64_t T, int64_t C, int iters, float eps_sk, float eps_rms,
                                float *Hpre, float *Hpost, float *Hres, float *u_save,
                                float *r_save, cudaStream_t s)
{
    MHC_PROF("k_pin_proj_fwd", s);
    launch_k(k_pin_proj_fwd, dim3(blocks(T, 64)), dim3(64), 0, s, x, W, alpha, b, T, C, iters,
             eps_sk, eps_rms, Hpre, Hpost, Hres, u_save, r_save);
    return cudaGetLastError();
}

namespace {
struct PinWs {
    float *du, *dz, *ga, *coef, *dHpre, *dHpost, *dHres;
};
PinWs carve_pin(void *ws, int64_t T)
{
    PinWs w;
    float *p = static_cast<float *>(ws);
    w.du = p;
    w.dz = w.du + T * PO;
    w.ga = w.dz + T * PO;
    w.coef = w.ga + T * 3;
    w.dHpre = w.coef + T;
    w.dHpost = w.dHpre + T * PN;
    w.dHres = w.dHpost + T * PN;
    return w;
}

// the proj backward from dH: per-token pass, dx (standalone or layer), dW, dalpha, db
cudaError_t pin_bwd_core(const float *dHpre, const float *dHpost, const float *dHres,
                         const bf16 *x, const float *W, const float *alpha, const float *b,
                         int64_t T, int64_t C, int iters, float eps_sk, float eps_rms,
                         const bf16 *dout, const bf16 *dy, const float *Hpre, const float *Hres,
                         bf16 *dx, float *dW, float *dalpha, float *db, const PinWs &w,
                         cudaStream_t s)
{
    const int64_t K = PN * C;
    {
        MHC_PROF("k_pin_bwd_token", s);
        launch_k(k_pin_bwd_token, dim3(blocks(T, 64)), dim3(64), 0, s, dHpre, dHpost, dHres, x,
                 W, alpha, b, T, C, iters, eps_sk, eps_rms, w.du, w.dz, w.ga, w.coef);
    }
    {
        MHC_PROF("k_pin_dx", s);
        launch_k(k_pin_dx, dim3(blocks(T * K, 256)), dim3(256), 0, s, x, W,
                 static_cast<const float *>(w.du), static_cast<const float *>(w.coef), T, C,
                 dout, dy, Hpre, Hres, dx);
    }
    {
        MHC_PROF("k_pin_dw", s);
        launch_k(k_pin_dw, dim3(blocks(K * PO, 256)), dim3(256), 0, s, x,
                 static_cast<const float *>(w.du), T, K, dW);
    }
    {
        MHC_PROF("k_pin_colfold", s);
        launch_k(k_pin_colfold, dim3(1), dim3(32), 0, s, static_cast<const float *>(w.dz), T, PO, db);
        launch_k(k_pin_colfold, dim3(1), dim3(32), 0, s, static_cast<const float *>(w.ga), T, 3,
                 dalpha);
    }
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_pin_proj_bwd(const float *dHpre, const float *dHpost, const float *dHres,
                                const bf16 *x, const float *W, const float *alpha, const float *b,
                                int64_t T, int64_t C, int iters, float eps_sk, float eps_rms,
                                bf16 *dx, float *dW, float *dalpha, float *db, void *ws,
                                cudaStream_t s)
{
    const PinWs w = carve_pin(ws, T);
    return pin_bwd_core(dHpre, dHpost, dHres, x, W, alpha, b, T, C, iters, eps_sk, eps_rms,
                        nullptr, nullptr, nullptr, nullptr, dx, dW, dalpha, db, w, s);
}

cudaError_t launch_pin_agg_fwd(const bf16 *x, const float *Hpre, bf16 *y, int64_t T, int64_t C,
                               cudaStream_t s)
{
    MHC_PROF("k_pin_agg_fwd", s);
    launch_k(k_pin_agg_fwd, dim3(blocks(T * C, 256)), dim3(256), 0, s, x, Hpre, T, C, y);
    return cudaGetLastError();
}

cudaError_t launch_pin_agg_bwd(const bf16 *dy, const bf16 *x, const float *Hpre, bf16 *dx,
                               float *dHpre, int64_t T, int64_t C, cudaStream_t s)
{
    {
        MHC_PROF("k_pin_agg_bwd_dx", s);
        launch_k(k_pin_agg_bwd_dx, dim3(blocks(T * PN * C, 256)), dim3(256), 0, s, dy, Hpre, T, C,
                 dx);
    }
    MHC_PROF("k_pin_tok_folds", s);
    launch_k(k_pin_tok_folds, dim3(blocks(T * 24)), dim3(128), 0, s, x,
             static_cast<const bf16 *>(nullptr), static_cast<const bf16 *>(nullptr),
             static_cast<const bf16 *>(nullptr), dy, T, C, static_cast<float *>(nullptr),
             static_cast<float *>(nullptr), dHpre);
    return cudaGetLastError();
}

cudaError_t launch_pin_post_fwd(const bf16 *res, const bf16 *f, const bf16 *bias,
                                const float *Hres, const float *Hpost, bf16 *out, int64_t T,
                                int64_t C, cudaStream_t s)
{
    MHC_PROF("k_pin_post_fwd", s);
    launch_k(k_pin_post_fwd, dim3(blocks(T * C, 256)), dim3(256), 0, s, res, f, bias, Hres, Hpost,
             T, C, out);
    return cudaGetLastError();
}

cudaError_t launch_pin_post_bwd(const bf16 *dout, const bf16 *res, const bf16 *f,
                                const bf16 *bias, const float *Hres, const float *Hpost,
                                bf16 *dres, bf16 *df, float *dbias, float *dHres, float *dHpost,
                                int64_t T, int64_t C, cudaStream_t s)
{
    {
        MHC_PROF("k_pin_post_bwd_elem", s);
        launch_k(k_pin_post_bwd_elem, dim3(blocks(T * C, 256)), dim3(256), 0, s, dout, Hres,
                 Hpost, T, C, dres, df);
    }
    {
        MHC_PROF("k_pin_tok_folds", s);
        launch_k(k_pin_tok_folds, dim3(blocks(T * 24)), dim3(128), 0, s, res, dout, f, bias,
                 static_cast<const bf16 *>(nullptr), T, C, dHres, dHpost,
                 static_cast<float *>(nullptr));
    }
    if (dbias) {
        MHC_PROF("k_pin_dbias", s);
        launch_k(k_pin_dbias, dim3(blocks(C, 128)), dim3(128), 0, s, dout, Hpost, T, C, dbias);
    }
    return cudaGetLastError();
}

cudaError_t launch_pin_layer_fwd(const bf16 *x, const float *W, const float *alpha,
                                 const float *b, const bf16 *f, const bf16 *bias, int64_t T,
                                 int64_t C, int iters, float eps_sk, float eps_rms, float *Hpre,
                                 float *Hpost, float *Hres, float *u_save, float *r_save, bf16 *y,
                                 bf16 *out, cudaStream_t s)
{
    cudaError_t e = launch_pin_proj_fwd(x, W, alpha, b, T, C, iters, eps_sk, eps_rms, Hpre, Hpost,
                                        Hres, u_save, r_save, s);
    if (e == cudaSuccess) e = launch_pin_agg_fwd(x, Hpre, y, T, C, s);
    if (e == cudaSuccess) e = launch_pin_post_fwd(x, f, bias, Hres, Hpost, out, T, C, s);
    return e;
}

cudaError_t launch_pin_layer_bwd(const bf16 *dout, const bf16 *dy, const bf16 *x, const float *W,
                                 const float *alpha, const float *b, const bf16 *f,
                                 const bf16 *bias, const float *Hpre, const float *Hpost,
                                 const float *Hres, int64_t T, int64_t C, int iters, float eps_sk,
                                 float eps_rms, bf16 *dx, bf16 *df, float *dW, float *dalpha,
                                 float *db, float *dbias, void *ws, cudaStream_t s)
{
    const PinWs w = carve_pin(ws, T);
    {
        MHC_PROF("k_pin_post_bwd_elem", s);
        launch_k(k_pin_post_bwd_elem, dim3(blocks(T * C, 256)), dim3(256), 0, s, dout, Hres, Hpost,
                 T, C, static_cast<bf16 *>(nullptr), df);
    }
    {
        MHC_PROF("k_pin_tok_folds", s);
        launch_k(k_pin_tok_folds, dim3(blocks(T * 24)), dim3(128), 0, s, x, dout, f, bias, dy, T, C,
                 w.dHres, w.dHpost, w.dHpre);
    }
    if (dbias) {
        MHC_PROF("k_pin_dbias", s);
        launch_k(k_pin_dbias, dim3(blocks(C, 128)), dim3(128), 0, s, dout, Hpost, T, C, dbias);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return pin_bwd_core(w.dHpre, w.dHpost, w.dHres, x, W, alpha, b, T, C, iters, eps_sk, eps_rms,
                        dout, dy, Hpre, Hres, dx, dW, dalpha, db, w, s);
}

}  // namespace mhc
