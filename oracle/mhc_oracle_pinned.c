/*
 * mHC residual-stream ops in fp32 with the pinned reduction order:
 * the reference the library's bit-reproducible mode is compared with,
 * bit for bit.
 *
 * TEST INFRASTRUCTURE ONLY (like mhc_oracle.c, whose fp64 definitions these
 * functions follow step for step).  The library never calls it.
 *
 * The numerical contract ([rlk] RL-Align/RL-Kernel PR #383, PR body,
 * "Numerical contract"): fp32 arithmetic, and only two reduction trees:
 * a serial ascending left fold for long reductions, and (a0 + a1) + (a2 + a3)
 * over the four streams.  Here, for n = 4:
 *   fold4(a0..a3)   = (a0 + a1) + (a2 + a3)
 *   fold(v_0..v_m)  = (((0 + v_0) + v_1) + ...) + v_m, ascending index
 * Every product is rounded to fp32 before it is added (no fused multiply-add;
 * this file is compiled with -ffp-contract=off), divisions and square roots
 * are the correctly rounded IEEE operations, and a bf16 output is the
 * round-to-nearest-even of its fp32 value.  The pages give the trees but not
 * the order of every non-reduction operation; the order used is the one
 * written below (it is the plain left-to-right reading of each formula).
 *
 * exp: the pages' operations need exp (sigmoid gates, Sinkhorn), and a
 * bitwise contract needs the same exp on every device, so pin_exp is written
 * here from its mathematics: Cody and Waite's argument reduction (x = n ln2
 * + r with ln2 split into a short high part and a low part, |r| <= ln2 / 2),
 * the Taylor series of e^r to degree 7 in Horner form with fused
 * multiply-adds (fmaf, an IEEE operation), and the exact scaling by 2^n.
 * Arguments are clamped to [-87, 88] so that the result stays a normal fp32
 * value.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define PN 4           /* the pinned trees are defined for four streams */
#define PO (PN * PN + 2 * PN)

static float fold4(float a0, float a1, float a2, float a3) { return (a0 + a1) + (a2 + a3); }

/* bf16 round-to-nearest-even of an fp32 value (finite inputs), as fp32 */
static float pin_bf16(float v)
{
    uint32_t u;
    memcpy(&u, &v, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    u &= 0xFFFF0000u;
    float r;
    memcpy(&r, &u, 4);
    return r;
}

float orc_pin_exp(float x)
{
    if (x > 88.0f) x = 88.0f;
    if (x < -87.0f) x = -87.0f;
    /* fp32 constants written exactly (hex): log2(e); ln2 split as a
     * 12-significant-bit high part (so n * ln2_hi is exact) and the fp32
     * value of the remainder; the Taylor coefficients 1/7!, 1/6!, 1/5!,
     * 1/4!, 1/3! rounded to fp32 */
    const float log2e = 0x1.715476p+0f;
    const float ln2_hi = 0x1.62e4p-1f;
    const float ln2_lo = 0x1.7f7d1cp-20f;
    const float n = rintf(x * log2e);
    float r = fmaf(-n, ln2_hi, x);
    r = fmaf(-n, ln2_lo, r);
    float p = 0x1.a01a02p-13f;
    p = fmaf(p, r, 0x1.6c16c2p-10f);
    p = fmaf(p, r, 0x1.111112p-7f);
    p = fmaf(p, r, 0x1.555556p-5f);
    p = fmaf(p, r, 0x1.555556p-3f);
    p = fmaf(p, r, 0.5f);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    const uint32_t bits = (uint32_t)((int)n + 127) << 23;
    float scale;
    memcpy(&scale, &bits, 4);
    return p * scale;
}

static float pin_sigmoid(float z) { return 1.0f / (1.0f + orc_pin_exp(-z)); }

/* Sinkhorn of one 4 x 4 matrix; trace as in mhc_oracle.c's sinkhorn_one. */
static void pin_sinkhorn(const float *z, int iters, float eps, float *P, float *trace)
{
    float A[PN * PN];
    for (int e = 0; e < PN * PN; ++e) A[e] = orc_pin_exp(z[e]);
    for (int k = 0; k < iters; ++k) {
        for (int i = 0; i < PN; ++i) {
            const float d = fold4(A[i * PN], A[i * PN + 1], A[i * PN + 2], A[i * PN + 3]) + eps;
            for (int j = 0; j < PN; ++j) A[i * PN + j] = A[i * PN + j] / d;
        }
        if (trace) memcpy(trace + (size_t)(2 * k) * PN * PN, A, sizeof(A));
        for (int j = 0; j < PN; ++j) {
            const float d = fold4(A[j], A[PN + j], A[2 * PN + j], A[3 * PN + j]) + eps;
            for (int i = 0; i < PN; ++i) A[i * PN + j] = A[i * PN + j] / d;
        }
        if (trace) memcpy(trace + (size_t)(2 * k + 1) * PN * PN, A, sizeof(A));
    }
    memcpy(P, A, sizeof(A));
}

/* Gradient of pin_sinkhorn (the steps of mhc_oracle.c's sinkhorn_bwd_one). */
static void pin_sinkhorn_bwd(const float *g_in, const float *z, int iters, float eps, float *dz,
                             float *trace)
{
    float P[PN * PN], E[PN * PN], G[PN * PN];
    pin_sinkhorn(z, iters, eps, P, trace);
    for (int e = 0; e < PN * PN; ++e) E[e] = orc_pin_exp(z[e]);
    memcpy(G, g_in, sizeof(G));
    for (int k = iters - 1; k >= 0; --k) {
        const float *Bk = trace + (size_t)(2 * k) * PN * PN;
        const float *Ak = trace + (size_t)(2 * k + 1) * PN * PN;
        const float *Ap = (k == 0) ? E : trace + (size_t)(2 * k - 1) * PN * PN;
        for (int j = 0; j < PN; ++j) {
            const float d = fold4(Bk[j], Bk[PN + j], Bk[2 * PN + j], Bk[3 * PN + j]) + eps;
            const float dot = fold4(G[j] * Ak[j], G[PN + j] * Ak[PN + j],
                                    G[2 * PN + j] * Ak[2 * PN + j], G[3 * PN + j] * Ak[3 * PN + j]);
            for (int i = 0; i < PN; ++i) G[i * PN + j] = (G[i * PN + j] - dot) / d;
        }
        for (int i = 0; i < PN; ++i) {
            const float *a = Ap + i * PN, *bb = Bk + i * PN;
            float *gg = G + i * PN;
            const float d = fold4(a[0], a[1], a[2], a[3]) + eps;
            const float dot = fold4(gg[0] * bb[0], gg[1] * bb[1], gg[2] * bb[2], gg[3] * bb[3]);
            for (int j = 0; j < PN; ++j) gg[j] = (gg[j] - dot) / d;
        }
    }
    for (int e = 0; e < PN * PN; ++e) dz[e] = G[e] * E[e];
}

int orc_pin_sinkhorn_fwd(const float *logits, float *P, int64_t M, int iters, float eps)
{
    for (int64_t m = 0; m < M; ++m) pin_sinkhorn(logits + m * PN * PN, iters, eps, P + m * PN * PN, 0);
    return 0;
}

int orc_pin_sinkhorn_bwd(const float *dP, const float *logits, float *dlogits, int64_t M,
                         int iters, float eps, float *trace_scratch)
{
    for (int64_t m = 0; m < M; ++m)
        pin_sinkhorn_bwd(dP + m * PN * PN, logits + m * PN * PN, iters, eps,
                         dlogits + m * PN * PN, trace_scratch);
    return 0;
}

/* ---- proj_rms_compute_h ------------------------------------------------ */

static float seg_alpha(const float *alpha, int o) { return o < PN ? alpha[0] : (o < 2 * PN ? alpha[1] : alpha[2]); }

/* one token: s = fold_k x^2, u[o] = fold_k x[k] W[k][o], q, r */
static void pin_proj_token(const float *xt, const float *W, int64_t K, float eps_rms, float *u,
                           float *q, float *r)
{
    float s = 0.0f;
    for (int o = 0; o < PO; ++o) u[o] = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
        const float xv = xt[k];
        s = s + xv * xv;
        for (int o = 0; o < PO; ++o) u[o] = u[o] + xv * W[k * PO + o];
    }
    *q = sqrtf(s / (float)K);
    *r = 1.0f / (*q + eps_rms);
}

/* z[o] = (alpha_seg r) u[o] + b[o] */
static void pin_logits(const float *u, float r, const float *alpha, const float *b, float *z)
{
    for (int o = 0; o < PO; ++o) z[o] = (seg_alpha(alpha, o) * r) * u[o] + b[o];
}

int orc_pin_proj_rms_compute_h_fwd(const float *x, const float *W, const float *alpha,
                                   const float *b, int64_t T, int64_t C, int iters, float eps_sk,
                                   float eps_rms, float *Hpre, float *Hpost, float *Hres,
                                   float *u_out, float *r_out)
{
    const int64_t K = PN * C;
    for (int64_t t = 0; t < T; ++t) {
        float u[PO], z[PO], q, r;
        pin_proj_token(x + t * K, W, K, eps_rms, u, &q, &r);
        pin_logits(u, r, alpha, b, z);
        for (int i = 0; i < PN; ++i) {
            Hpre[t * PN + i] = pin_sigmoid(z[i]);
            Hpost[t * PN + i] = 2.0f * pin_sigmoid(z[PN + i]);
        }
        pin_sinkhorn(z + 2 * PN, iters, eps_sk, Hres + t * PN * PN, 0);
        if (u_out) memcpy(u_out + t * PO, u, sizeof(u));
        if (r_out) r_out[t] = r;
    }
    return 0;
}

/* Per-token backward quantities (from the fp64 oracle's steps):
 *   dz_pre = (dH_pre s) (1 - s), dz_post = ((2 dH_post) s) (1 - s),
 *   dz_res = Sinkhorn backward, g_seg = fold_{o in seg} dz[o] u[o],
 *   ga_seg = g_seg r, dr = fold_seg alpha_seg g_seg,
 *   du[o] = (alpha_seg r) dz[o], coef = ((-dr r) r) / (K q)  (0 when q = 0). */
static void pin_bwd_token(const float *dHpre, const float *dHpost, const float *dHres,
                          const float *u, float q, float r, const float *alpha, const float *b,
                          int64_t K, int iters, float eps_sk, float *trace, float *dz, float *du,
                          float *ga, float *coef)
{
    float z[PO];
    pin_logits(u, r, alpha, b, z);
    for (int i = 0; i < PN; ++i) {
        const float sp = pin_sigmoid(z[i]), so = pin_sigmoid(z[PN + i]);
        dz[i] = (dHpre[i] * sp) * (1.0f - sp);
        dz[PN + i] = ((2.0f * dHpost[i]) * so) * (1.0f - so);
    }
    pin_sinkhorn_bwd(dHres, z + 2 * PN, iters, eps_sk, dz + 2 * PN, trace);
    float g[3] = {0.0f, 0.0f, 0.0f};
    for (int o = 0; o < PO; ++o) {
        const int sg = o < PN ? 0 : (o < 2 * PN ? 1 : 2);
        g[sg] = g[sg] + dz[o] * u[o];
    }
    float dr = 0.0f;
    for (int s = 0; s < 3; ++s) {
        ga[s] = g[s] * r;
        dr = dr + alpha[s] * g[s];
    }
    for (int o = 0; o < PO; ++o) du[o] = (seg_alpha(alpha, o) * r) * dz[o];
    *coef = (q > 0.0f) ? ((-dr * r) * r) / ((float)K * q) : 0.0f;
}

/* dx_proj[k] = fold_o du[o] W[k][o] + coef x[k] */
static float pin_dx_proj(const float *du, const float *Wk, float coef, float xk)
{
    float acc = 0.0f;
    for (int o = 0; o < PO; ++o) acc = acc + du[o] * Wk[o];
    return acc + coef * xk;
}

/* Backward of proj_rms_compute_h (standalone op).  The sums over tokens
 * (dW, dalpha, db) fold in ascending t.  Scratch: T * (2 * PO + 4) floats
 * plus (2 iters + 1) 16-float trace matrices. */
int orc_pin_proj_rms_compute_h_bwd(const float *dHpre, const float *dHpost, const float *dHres,
                                   const float *x, const float *W, const float *alpha,
                                   const float *b, int64_t T, int64_t C, int iters,
                                   float eps_sk, float eps_rms, float *dx, float *dW,
                                   float *dalpha, float *db, float *scratch, float *trace)
{
    const int64_t K = PN * C;
    float *du_all = scratch, *dz_all = scratch + T * PO, *ga_all = scratch + 2 * T * PO;
    for (int64_t t = 0; t < T; ++t) {
        float u[PO], q, r, coef;
        const float *xt = x + t * K;
        pin_proj_token(xt, W, K, eps_rms, u, &q, &r);
        pin_bwd_token(dHpre + t * PN, dHpost + t * PN, dHres + t * PN * PN, u, q, r, alpha, b, K,
                      iters, eps_sk, trace, dz_all + t * PO, du_all + t * PO, ga_all + t * 3, &coef);
        for (int64_t k = 0; k < K; ++k)
            dx[t * K + k] = pin_bf16(pin_dx_proj(du_all + t * PO, W + k * PO, coef, xt[k]));
    }
    for (int64_t k = 0; k < K; ++k)
        for (int o = 0; o < PO; ++o) {
            float acc = 0.0f;
            for (int64_t t = 0; t < T; ++t) acc = acc + x[t * K + k] * du_all[t * PO + o];
            dW[k * PO + o] = acc;
        }
    for (int s = 0; s < 3; ++s) {
        float acc = 0.0f;
        for (int64_t t = 0; t < T; ++t) acc = acc + ga_all[t * 3 + s];
        dalpha[s] = acc;
    }
    for (int o = 0; o < PO; ++o) {
        float acc = 0.0f;
        for (int64_t t = 0; t < T; ++t) acc = acc + dz_all[t * PO + o];
        db[o] = acc;
    }
    return 0;
}

/* ---- h_aggregate and h_post_bda ---------------------------------------- */

int orc_pin_h_aggregate_fwd(const float *x, const float *Hpre, int64_t T, int64_t C, float *y)
{
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < C; ++c) {
            const float *xt = x + t * PN * C + c, *h = Hpre + t * PN;
            y[t * C + c] = pin_bf16(fold4(h[0] * xt[0], h[1] * xt[C], h[2] * xt[2 * C], h[3] * xt[3 * C]));
        }
    return 0;
}

/* dx[t][i][c] = H_pre[t][i] dy[t][c] (bf16); dH_pre[t][i] = fold_c dy x */
int orc_pin_h_aggregate_bwd(const float *dy, const float *x, const float *Hpre, int64_t T,
                            int64_t C, float *dx, float *dHpre)
{
    for (int64_t t = 0; t < T; ++t)
        for (int i = 0; i < PN; ++i) {
            float acc = 0.0f;
            for (int64_t c = 0; c < C; ++c) {
                const float d = dy[t * C + c];
                if (dx) dx[(t * PN + i) * C + c] = pin_bf16(Hpre[t * PN + i] * d);
                acc = acc + d * x[(t * PN + i) * C + c];
            }
            dHpre[t * PN + i] = acc;
        }
    return 0;
}

/* out[t][i][c] = fold4_j(H_res[t][j][i] x[t][j][c]) + H_post[t][i] (f[t][c] + bias[c]) */
int orc_pin_h_post_bda_fwd(const float *res, const float *f, const float *bias, const float *Hres,
                           const float *Hpost, int64_t T, int64_t C, float *out)
{
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < C; ++c) {
            const float g = f[t * C + c] + (bias ? bias[c] : 0.0f);
            const float *xr = res + t * PN * C + c, *hr = Hres + t * PN * PN;
            for (int i = 0; i < PN; ++i) {
                const float m = fold4(hr[i] * xr[0], hr[PN + i] * xr[C], hr[2 * PN + i] * xr[2 * C],
                                      hr[3 * PN + i] * xr[3 * C]);
                out[(t * PN + i) * C + c] = pin_bf16(m + Hpost[t * PN + i] * g);
            }
        }
    return 0;
}

/* dres[t][j][c] = fold4_i(H_res[j][i] dout[i][c]) (bf16), dfv = fold4_i(H_post[i] dout[i][c]),
 * df = bf16(dfv), dH_res[t][j][i] = fold_c x[j][c] dout[i][c],
 * dH_post[t][i] = fold_c dout[i][c] (f[c] + bias[c]), dbias[c] = fold_t dfv[t][c]. */
int orc_pin_h_post_bda_bwd(const float *dout, const float *res, const float *f, const float *bias,
                           const float *Hres, const float *Hpost, int64_t T, int64_t C,
                           float *dres, float *df, float *dbias, float *dHres, float *dHpost)
{
    for (int64_t c = 0; c < C; ++c) if (dbias) dbias[c] = 0.0f;
    for (int64_t t = 0; t < T; ++t) {
        const float *hr = Hres + t * PN * PN, *hp = Hpost + t * PN;
        const float *dt = dout + t * PN * C, *xt = res + t * PN * C;
        for (int64_t c = 0; c < C; ++c) {
            const float dfv = fold4(hp[0] * dt[c], hp[1] * dt[C + c], hp[2] * dt[2 * C + c],
                                    hp[3] * dt[3 * C + c]);
            if (df) df[t * C + c] = pin_bf16(dfv);
            if (dbias) dbias[c] = dbias[c] + dfv;
            if (dres)
                for (int j = 0; j < PN; ++j)
                    dres[(t * PN + j) * C + c] = pin_bf16(fold4(
                        hr[j * PN] * dt[c], hr[j * PN + 1] * dt[C + c], hr[j * PN + 2] * dt[2 * C + c],
                        hr[j * PN + 3] * dt[3 * C + c]));
        }
        for (int j = 0; j < PN; ++j)
            for (int i = 0; i < PN; ++i) {
                float acc = 0.0f;
                for (int64_t c = 0; c < C; ++c) acc = acc + xt[j * C + c] * dt[i * C + c];
                dHres[(t * PN + j) * PN + i] = acc;
            }
        for (int i = 0; i < PN; ++i) {
            float acc = 0.0f;
            for (int64_t c = 0; c < C; ++c)
                acc = acc + dt[i * C + c] * (f[t * C + c] + (bias ? bias[c] : 0.0f));
            dHpost[t * PN + i] = acc;
        }
    }
    return 0;
}

/* ---- the layer backward's residual gradient ---------------------------- */

/* The layer backward in pinned order: the post_bda and aggregate sums above,
 * the proj backward with those dH, and
 *   dx[t][j][c] = bf16((fold4_i(H_res[j][i] dout[i][c]) + H_pre[j] dy[c])
 *                      + (fold_o du[o] W[k][o] + coef x[k])),  k = j C + c.
 * The per-token u and r are recomputed from x (the pinned forward's values).
 * Scratch: T * (2 * PO + 4 + 2 * PN + PN * PN) floats plus a trace. */
int orc_pin_layer_bwd(const float *dout, const float *dy, const float *x, const float *W,
                      const float *alpha, const float *b, const float *f, const float *bias,
                      const float *Hpre, const float *Hpost, const float *Hres, int64_t T,
                      int64_t C, int iters, float eps_sk, float eps_rms, float *dx, float *df,
                      float *dW, float *dalpha, float *db, float *dbias, float *scratch,
                      float *trace)
{
    const int64_t K = PN * C;
    float *du_all = scratch, *dz_all = scratch + T * PO, *ga_all = scratch + 2 * T * PO;
    float *dHp = ga_all + 3 * T, *dHq = dHp + PN * T, *dHr = dHq + PN * T;
    float *coef_all = dHr + PN * PN * T;
    orc_pin_h_post_bda_bwd(dout, x, f, bias, Hres, Hpost, T, C, 0, df, dbias, dHr, dHq);
    orc_pin_h_aggregate_bwd(dy, x, Hpre, T, C, 0, dHp);
    for (int64_t t = 0; t < T; ++t) {
        float u[PO], q, r;
        pin_proj_token(x + t * K, W, K, eps_rms, u, &q, &r);
        pin_bwd_token(dHp + t * PN, dHq + t * PN, dHr + t * PN * PN, u, q, r, alpha, b, K, iters,
                      eps_sk, trace, dz_all + t * PO, du_all + t * PO, ga_all + t * 3,
                      coef_all + t);
        const float *hr = Hres + t * PN * PN, *dt = dout + t * PN * C;
        for (int j = 0; j < PN; ++j)
            for (int64_t c = 0; c < C; ++c) {
                const int64_t k = j * C + c;
                const float dres = fold4(hr[j * PN] * dt[c], hr[j * PN + 1] * dt[C + c],
                                         hr[j * PN + 2] * dt[2 * C + c], hr[j * PN + 3] * dt[3 * C + c]);
                const float dagg = Hpre[t * PN + j] * dy[t * C + c];
                const float dproj = pin_dx_proj(du_all + t * PO, W + k * PO, coef_all[t], x[t * K + k]);
                dx[t * K + k] = pin_bf16((dres + dagg) + dproj);
            }
    }
    for (int64_t k = 0; k < K; ++k)
        for (int o = 0; o < PO; ++o) {
            float acc = 0.0f;
            for (int64_t t = 0; t < T; ++t) acc = acc + x[t * K + k] * du_all[t * PO + o];
            dW[k * PO + o] = acc;
        }
    for (int s = 0; s < 3; ++s) {
        float acc = 0.0f;
        for (int64_t t = 0; t < T; ++t) acc = acc + ga_all[t * 3 + s];
        dalpha[s] = acc;
    }
    for (int o = 0; o < PO; ++o) {
        float acc = 0.0f;
        for (int64_t t = 0; t < T; ++t) acc = acc + dz_all[t * PO + o];
        db[o] = acc;
    }
    return 0;
}
