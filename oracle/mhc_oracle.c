/*
 * mHC residual-stream ops: plain CPU fp64 oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * definition that the CUDA library is checked against.  Only the tests, the
 * smoke check and the benchmark's CPU-baseline leg may load it; the library
 * never calls it and shares no code with it.
 *
 * Every function is the plain definition: double accumulators, loops in
 * ascending index order, no blocking or fusion.  Every argument is double:
 * the caller passes the exact values the GPU receives (a bf16 or fp32 value
 * converts to double without rounding), so finite differences can also
 * perturb any input.  OpenMP only splits independent tokens
 * (or independent output rows of a sum over tokens); no reduction changes
 * order with the thread count.
 *
 * Sources (web pages; see the header of each function for the part used):
 *  [rwkv]  rwkv-ops 0.6.1, rwkv_ops/mhc_kernel/jax_kernel/mhu_ffi.cu
 *          (XLA-FFI handlers SinkhornFwdHost/BwdHost, RMSNormFwd/BwdHost,
 *          StreamAggregateFwd/Bwd, MhcPostOpFwd/BwdHost, MhcPreOpFwd/BwdHost)
 *  [mcore] Megatron-Core API docs, core.fusions.fused_mhc_kernels
 *          (fused_sinkhorn, fused_h_aggregate, fused_h_post_bda,
 *          fused_proj_rms_compute_h, _torch_proj_rms_compute_h,
 *          _torch_h_post_bda_bwd, FusedHAggregate, FusedHPostBDA)
 *  [rlk]   RL-Align/RL-Kernel PR #383, "[DSv4][P1-S0] Start kit for the P1
 *          work package (mHC + RMSNorm)": review of oracle.py (RMS backward
 *          zero-row guard), the follow-up commit on Megatron's three alpha
 *          scalars and sqrt(s/K), and the PR body's task list.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - RMS of the flattened residual: r = 1/(sqrt(s/K) + eps_rms), eps outside
 *    the root ([rlk] review: forward r = 1/(q+eps), backward -r^2 x/(K q)).
 *  - z = alpha_seg * r * u + b with u = x.W, segments pre|post|res, res
 *    row-major ([rlk] commit: three scalars over PRE/POST/COMB).
 *  - H_pre = sigmoid(z_pre), H_post = 2 sigmoid(z_post) ([rwkv] MhcPreOpFwd
 *    output comments), H_res = Sinkhorn(exp(z_res)).
 *  - Sinkhorn: plain exp, then `iters` times: every row divided by (its sum +
 *    eps), then every column divided by (its sum + eps).  Backward is the
 *    exact gradient of that unrolled map ([rwkv] SinkhornBwdHost takes the
 *    iteration count and the raw input).
 *  - post_bda: out[i] = sum_j H_res[j][i] x[j] + H_post[i] (f + bias)
 *    ([mcore] "H_res.T @ residual + H_post * (x + bias)"), dropout p = 0.
 *  - Standalone RMSNorm: y = x / sqrt(mean(x^2) + eps), no weight ([rwkv]
 *    RMSNormFwdHost has only input, output and eps).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_MAX_N 16

static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* ------------------------------------------------------------------------ */
/* Sinkhorn-Knopp ([rwkv] SinkhornFwdHost / SinkhornBwdHost; [mcore]        */
/* fused_sinkhorn "projection to doubly stochastic matrix").                 */
/* ------------------------------------------------------------------------ */

/* Forward on one n x n matrix of logits z (row-major).  If `trace` is not
 * NULL it receives the 2*iters intermediate matrices: trace[2k] = after the
 * row step of iteration k, trace[2k+1] = after its column step. */
static void sinkhorn_one(const double *z, int n, int iters, double eps,
                         double *P, double *trace)
{
    double A[ORC_MAX_N * ORC_MAX_N];
    for (int e = 0; e < n * n; ++e) A[e] = exp(z[e]);
    for (int k = 0; k < iters; ++k) {
        for (int i = 0; i < n; ++i) {
            double s = 0.0;
            for (int j = 0; j < n; ++j) s += A[i * n + j];
            for (int j = 0; j < n; ++j) A[i * n + j] /= (s + eps);
        }
        if (trace) memcpy(trace + (size_t)(2 * k) * n * n, A, sizeof(double) * n * n);
        for (int j = 0; j < n; ++j) {
            double s = 0.0;
            for (int i = 0; i < n; ++i) s += A[i * n + j];
            for (int i = 0; i < n; ++i) A[i * n + j] /= (s + eps);
        }
        if (trace) memcpy(trace + (size_t)(2 * k + 1) * n * n, A, sizeof(double) * n * n);
    }
    memcpy(P, A, sizeof(double) * n * n);
}

/* Exact gradient of sinkhorn_one with respect to z, given dL/dP = g.
 * A step X -> Y with Y[i][j] = X[i][j] / d_i, d_i = sum_j X[i][j] + eps, has
 * dL/dX[i][j] = (dL/dY[i][j] - sum_j' dL/dY[i][j'] Y[i][j']) / d_i; the
 * column step is the same with rows and columns exchanged.  The first
 * matrix is exp(z), so dL/dz = dL/dA0 * exp(z). */
static void sinkhorn_bwd_one(const double *g_in, const double *z, int n, int iters,
                             double eps, double *dz, double *trace)
{
    double P[ORC_MAX_N * ORC_MAX_N], E[ORC_MAX_N * ORC_MAX_N];
    double G[ORC_MAX_N * ORC_MAX_N];
    sinkhorn_one(z, n, iters, eps, P, trace);
    for (int e = 0; e < n * n; ++e) E[e] = exp(z[e]);
    memcpy(G, g_in, sizeof(double) * n * n);
    for (int k = iters - 1; k >= 0; --k) {
        const double *Bk = trace + (size_t)(2 * k) * n * n;     /* after row step */
        const double *Ak = trace + (size_t)(2 * k + 1) * n * n; /* after col step */
        const double *Aprev = (k == 0) ? E : trace + (size_t)(2 * k - 1) * n * n;
        /* column step backward: Ak = Bk / (colsum(Bk) + eps) */
        for (int j = 0; j < n; ++j) {
            double cs = 0.0, dot = 0.0;
            for (int i = 0; i < n; ++i) cs += Bk[i * n + j];
            for (int i = 0; i < n; ++i) dot += G[i * n + j] * Ak[i * n + j];
            for (int i = 0; i < n; ++i) G[i * n + j] = (G[i * n + j] - dot) / (cs + eps);
        }
        /* row step backward: Bk = Aprev / (rowsum(Aprev) + eps) */
        for (int i = 0; i < n; ++i) {
            double rs = 0.0, dot = 0.0;
            for (int j = 0; j < n; ++j) rs += Aprev[i * n + j];
            for (int j = 0; j < n; ++j) dot += G[i * n + j] * Bk[i * n + j];
            for (int j = 0; j < n; ++j) G[i * n + j] = (G[i * n + j] - dot) / (rs + eps);
        }
    }
    for (int e = 0; e < n * n; ++e) dz[e] = G[e] * E[e];
}

int orc_sinkhorn_fwd(const double *logits, double *P, int64_t M, int n, int iters, double eps)
{
    if (n < 1 || n > ORC_MAX_N || iters < 0) return 1;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        double z[ORC_MAX_N * ORC_MAX_N];
        for (int e = 0; e < n * n; ++e) z[e] = logits[m * n * n + e];
        sinkhorn_one(z, n, iters, eps, P + m * n * n, NULL);
    }
    return 0;
}

int orc_sinkhorn_bwd(const double *dP, const double *logits, double *dlogits, int64_t M,
                     int n, int iters, double eps)
{
    if (n < 1 || n > ORC_MAX_N || iters < 0) return 1;
    const size_t trace_len = (size_t)(2 * iters + 1) * n * n;
    double *traces = (double *)malloc(sizeof(double) * trace_len * (size_t)(M > 0 ? M : 1));
    if (!traces) return 2;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        double z[ORC_MAX_N * ORC_MAX_N], g[ORC_MAX_N * ORC_MAX_N];
        for (int e = 0; e < n * n; ++e) {
            z[e] = logits[m * n * n + e];
            g[e] = dP[m * n * n + e];
        }
        sinkhorn_bwd_one(g, z, n, iters, eps, dlogits + m * n * n, traces + (size_t)m * trace_len);
    }
    free(traces);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* proj_rms_compute_h ([mcore] fused_proj_rms_compute_h /                    */
/* _torch_proj_rms_compute_h(x, weight, alpha_pre, alpha_post, alpha_res,    */
/* bias, n, eps, compute_h_eps); [rlk] fp32_gemm_rms forward and backward).  */
/* ------------------------------------------------------------------------ */

static double seg_alpha(const double *alpha, int n, int o)
{
    if (o < n) return alpha[0];
    if (o < 2 * n) return alpha[1];
    return alpha[2];
}

/* One token: s = sum x^2, q = sqrt(s/K), r = 1/(q + eps_rms), u = x.W. */
static void proj_rms_token(const double *xt, const double *W, int64_t K, int O,
                           double *u, double *q_out, double *r_out, double eps_rms)
{
    double s = 0.0;
    for (int o = 0; o < O; ++o) u[o] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double xv = xt[k];
        s += xv * xv;
        for (int o = 0; o < O; ++o) u[o] += xv * W[k * O + o];
    }
    double q = sqrt(s / (double)K);
    *q_out = q;
    *r_out = 1.0 / (q + eps_rms);
}

/* compute_h on one token's logits z[O]: gates and Sinkhorn. */
static void compute_h_token(const double *z, int n, int iters, double eps_sk,
                            double *Hpre, double *Hpost, double *Hres)
{
    for (int i = 0; i < n; ++i) {
        Hpre[i] = sigmoid(z[i]);
        Hpost[i] = 2.0 * sigmoid(z[n + i]);
    }
    sinkhorn_one(z + 2 * n, n, iters, eps_sk, Hres, NULL);
}

int orc_proj_rms_compute_h_fwd(const double *x, const double *W, const double *alpha,
                               const double *b, int64_t T, int n, int64_t C, int iters,
                               double eps_sk, double eps_rms, double *Hpre, double *Hpost,
                               double *Hres, double *u_out, double *r_out)
{
    if (n < 1 || n > ORC_MAX_N) return 1;
    const int O = n * n + 2 * n;
    const int64_t K = (int64_t)n * C;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double u[ORC_MAX_N * ORC_MAX_N + 2 * ORC_MAX_N], z[ORC_MAX_N * ORC_MAX_N + 2 * ORC_MAX_N];
        double q, r;
        proj_rms_token(x + t * K, W, K, O, u, &q, &r, eps_rms);
        for (int o = 0; o < O; ++o) z[o] = seg_alpha(alpha, n, o) * r * u[o] + b[o];
        compute_h_token(z, n, iters, eps_sk, Hpre + t * n, Hpost + t * n, Hres + t * n * n);
        if (u_out)
            for (int o = 0; o < O; ++o) u_out[t * O + o] = u[o];
        if (r_out) r_out[t] = r;
    }
    return 0;
}

/* Backward of proj_rms_compute_h.  Per token (recomputing the forward):
 *   dz_pre  = dH_pre  * s(1-s)          with s = sigmoid(z_pre)
 *   dz_post = dH_post * 2 s(1-s)        with s = sigmoid(z_post)
 *   dz_res  = Sinkhorn backward of dH_res
 *   dalpha_seg += sum_{o in seg} dz[o] r u[o];   db[o] += dz[o]
 *   du[o] = alpha_seg r dz[o];   dr = sum_o dz[o] alpha_seg u[o]
 *   dx[k] = sum_o du[o] W[k][o] + dr * (-r^2 x[k] / (K q))   (0 when q == 0,
 *           [rlk] review: the gradient of an all-zero row is 0)
 *   dW[k][o] = sum_t x[t][k] du[t][o]
 * Any of dx, dW, dalpha, db may be NULL.  Sums over tokens run in ascending t. */
int orc_proj_rms_compute_h_bwd(const double *dHpre, const double *dHpost, const double *dHres,
                               const double *x, const double *W, const double *alpha,
                               const double *b, int64_t T, int n, int64_t C, int iters,
                               double eps_sk, double eps_rms, double *dx, double *dW,
                               double *dalpha, double *db)
{
    if (n < 1 || n > ORC_MAX_N) return 1;
    const int O = n * n + 2 * n;
    const int64_t K = (int64_t)n * C;
    double *du_all = (double *)malloc(sizeof(double) * (size_t)T * O);
    double *ga_all = (double *)malloc(sizeof(double) * (size_t)T * 3); /* per-token dalpha terms */
    double *dz_all = (double *)malloc(sizeof(double) * (size_t)T * O);
    if (!du_all || !ga_all || !dz_all) {
        free(du_all); free(ga_all); free(dz_all);
        return 2;
    }
    const size_t trace_len = (size_t)(2 * iters + 1) * n * n;
    double *traces = (double *)malloc(sizeof(double) * trace_len * (size_t)(T > 0 ? T : 1));
    int rc = traces ? 0 : 2;
    if (rc == 0) {
#pragma omp parallel for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            double *trace = traces + (size_t)t * trace_len;
            double u[ORC_MAX_N * ORC_MAX_N + 2 * ORC_MAX_N], z[ORC_MAX_N * ORC_MAX_N + 2 * ORC_MAX_N];
            double dz[ORC_MAX_N * ORC_MAX_N + 2 * ORC_MAX_N], g[ORC_MAX_N * ORC_MAX_N];
            double q, r;
            const double *xt = x + t * K;
            proj_rms_token(xt, W, K, O, u, &q, &r, eps_rms);
            for (int o = 0; o < O; ++o) z[o] = seg_alpha(alpha, n, o) * r * u[o] + b[o];
            for (int i = 0; i < n; ++i) {
                double sp = sigmoid(z[i]);
                double so = sigmoid(z[n + i]);
                dz[i] = dHpre[t * n + i] * sp * (1.0 - sp);
                dz[n + i] = dHpost[t * n + i] * 2.0 * so * (1.0 - so);
            }
            for (int e = 0; e < n * n; ++e) g[e] = dHres[t * n * n + e];
            sinkhorn_bwd_one(g, z + 2 * n, n, iters, eps_sk, dz + 2 * n, trace);
            double ga[3] = {0.0, 0.0, 0.0};
            double dr = 0.0;
            for (int o = 0; o < O; ++o) {
                int sgi = (o < n) ? 0 : (o < 2 * n ? 1 : 2);
                ga[sgi] += dz[o] * r * u[o];
                dr += dz[o] * seg_alpha(alpha, n, o) * u[o];
                du_all[t * O + o] = seg_alpha(alpha, n, o) * r * dz[o];
                dz_all[t * O + o] = dz[o];
            }
            for (int s = 0; s < 3; ++s) ga_all[t * 3 + s] = ga[s];
            if (dx) {
                double coef = (q > 0.0) ? dr * (-(r * r) / ((double)K * q)) : 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    double acc = 0.0;
                    for (int o = 0; o < O; ++o) acc += du_all[t * O + o] * W[k * O + o];
                    dx[t * K + k] = acc + coef * xt[k];
                }
            }
        }
    }
    free(traces);
    if (rc == 0 && dW) {
#pragma omp parallel for schedule(static)
        for (int64_t k = 0; k < K; ++k) {
            double acc[ORC_MAX_N * ORC_MAX_N + 2 * ORC_MAX_N];
            for (int o = 0; o < O; ++o) acc[o] = 0.0;
            for (int64_t t = 0; t < T; ++t) {
                double xv = x[t * K + k];
                for (int o = 0; o < O; ++o) acc[o] += xv * du_all[t * O + o];
            }
            for (int o = 0; o < O; ++o) dW[k * O + o] = acc[o];
        }
    }
    if (rc == 0 && dalpha) {
        for (int s = 0; s < 3; ++s) dalpha[s] = 0.0;
        for (int64_t t = 0; t < T; ++t)
            for (int s = 0; s < 3; ++s) dalpha[s] += ga_all[t * 3 + s];
    }
    if (rc == 0 && db) {
        for (int o = 0; o < O; ++o) db[o] = 0.0;
        for (int64_t t = 0; t < T; ++t)
            for (int o = 0; o < O; ++o) db[o] += dz_all[t * O + o];
    }
    free(du_all); free(ga_all); free(dz_all);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* h_aggregate ([mcore] fused_h_aggregate, FusedHAggregate, _torch_h_        */
/* aggregate_bwd; [rwkv] StreamAggregateFwd/Bwd).                            */
/*   y[t][c] = sum_i H_pre[t][i] x[t][i][c]                                   */
/*   dx[t][i][c] = H_pre[t][i] dy[t][c];  dH_pre[t][i] = sum_c dy[t][c] x[t][i][c] */
/* ------------------------------------------------------------------------ */

int orc_h_aggregate_fwd(const double *x, const double *Hpre, int64_t T, int n, int64_t C,
                        double *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < C; ++c) {
            double acc = 0.0;
            for (int i = 0; i < n; ++i) acc += Hpre[t * n + i] * x[(t * n + i) * C + c];
            y[t * C + c] = acc;
        }
    return 0;
}

int orc_h_aggregate_bwd(const double *dy, const double *x, const double *Hpre, int64_t T,
                        int n, int64_t C, double *dx, double *dHpre)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int i = 0; i < n; ++i) {
            double acc = 0.0;
            for (int64_t c = 0; c < C; ++c) {
                double g = dy[t * C + c];
                if (dx) dx[(t * n + i) * C + c] = Hpre[t * n + i] * g;
                acc += g * x[(t * n + i) * C + c];
            }
            if (dHpre) dHpre[t * n + i] = acc;
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* h_post_bda ([mcore] fused_h_post_bda "H_res.T @ residual + H_post *       */
/* (x + bias)", _torch_h_post_bda_bwd returning five grads; [rwkv]           */
/* MhcPostOpFwdHost / MhcPostOpBwdHost).                                     */
/*   out[t][i][c] = sum_j H_res[t][j][i] res[t][j][c] + H_post[t][i] (f[t][c] + bias[c]) */
/* ------------------------------------------------------------------------ */

int orc_h_post_bda_fwd(const double *res, const double *f, const double *bias,
                       const double *Hres, const double *Hpost, int64_t T, int n, int64_t C,
                       double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int i = 0; i < n; ++i)
            for (int64_t c = 0; c < C; ++c) {
                double acc = 0.0;
                for (int j = 0; j < n; ++j)
                    acc += Hres[(t * n + j) * n + i] * res[(t * n + j) * C + c];
                double fb = f[t * C + c] + (bias ? bias[c] : 0.0);
                out[(t * n + i) * C + c] = acc + Hpost[t * n + i] * fb;
            }
    return 0;
}

/*   dres[t][j][c]  = sum_i H_res[t][j][i] dout[t][i][c]
 *   dH_res[t][j][i] = sum_c res[t][j][c] dout[t][i][c]
 *   dH_post[t][i]  = sum_c dout[t][i][c] (f[t][c] + bias[c])
 *   df[t][c]       = sum_i H_post[t][i] dout[t][i][c]
 *   dbias[c]       = sum_t df[t][c]          (ascending t)
 * Any output may be NULL. */
int orc_h_post_bda_bwd(const double *dout, const double *res, const double *f,
                       const double *bias, const double *Hres, const double *Hpost,
                       int64_t T, int n, int64_t C, double *dres, double *df, double *dbias,
                       double *dHres, double *dHpost)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        for (int j = 0; j < n; ++j) {
            for (int i = 0; i < n; ++i) {
                double acc = 0.0;
                for (int64_t c = 0; c < C; ++c)
                    acc += res[(t * n + j) * C + c] * dout[(t * n + i) * C + c];
                if (dHres) dHres[(t * n + j) * n + i] = acc;
            }
            if (dres)
                for (int64_t c = 0; c < C; ++c) {
                    double acc = 0.0;
                    for (int i = 0; i < n; ++i)
                        acc += Hres[(t * n + j) * n + i] * dout[(t * n + i) * C + c];
                    dres[(t * n + j) * C + c] = acc;
                }
        }
        for (int i = 0; i < n; ++i) {
            double acc = 0.0;
            for (int64_t c = 0; c < C; ++c) {
                double fb = f[t * C + c] + (bias ? bias[c] : 0.0);
                acc += dout[(t * n + i) * C + c] * fb;
            }
            if (dHpost) dHpost[t * n + i] = acc;
        }
        if (df)
            for (int64_t c = 0; c < C; ++c) {
                double acc = 0.0;
                for (int i = 0; i < n; ++i) acc += Hpost[t * n + i] * dout[(t * n + i) * C + c];
                df[t * C + c] = acc;
            }
    }
    if (dbias) {
#pragma omp parallel for schedule(static)
        for (int64_t c = 0; c < C; ++c) {
            double acc = 0.0;
            for (int64_t t = 0; t < T; ++t) {
                double g = 0.0;
                for (int i = 0; i < n; ++i) g += Hpost[t * n + i] * dout[(t * n + i) * C + c];
                acc += g;
            }
            dbias[c] = acc;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Standalone RMSNorm ([rwkv] RMSNormFwdHost / RMSNormBwdHost: bf16 [N, C],  */
/* eps, no weight).                                                          */
/*   rho = 1 / sqrt(sum_c x^2 / C + eps);  y = x rho                          */
/*   dx = rho dy - rho^3 x (sum_c dy x) / C                                   */
/* ------------------------------------------------------------------------ */

int orc_rmsnorm_fwd(const double *x, int64_t rows, int64_t cols, double eps, double *y,
                    double *rstd)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double s = 0.0;
        for (int64_t c = 0; c < cols; ++c) {
            double v = x[r * cols + c];
            s += v * v;
        }
        double rho = 1.0 / sqrt(s / (double)cols + eps);
        if (rstd) rstd[r] = rho;
        if (y)
            for (int64_t c = 0; c < cols; ++c) y[r * cols + c] = x[r * cols + c] * rho;
    }
    return 0;
}

int orc_rmsnorm_bwd(const double *dy, const double *x, int64_t rows, int64_t cols, double eps,
                    double *dx)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double s = 0.0, d = 0.0;
        for (int64_t c = 0; c < cols; ++c) {
            double v = x[r * cols + c];
            s += v * v;
            d += dy[r * cols + c] * v;
        }
        double rho = 1.0 / sqrt(s / (double)cols + eps);
        for (int64_t c = 0; c < cols; ++c)
            dx[r * cols + c] = rho * dy[r * cols + c] -
                               rho * rho * rho * x[r * cols + c] * d / (double)cols;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* h_aggregate with one static weight vector ([rwkv] StreamAggregateFwd/Bwd  */
/* with per_token = false: H_pre is [n] instead of [B, T, n], and d_H_pre is */
/* [n]).                                                                     */
/*   y[t][c] = sum_i H_pre[i] x[t][i][c]                                      */
/*   dx[t][i][c] = H_pre[i] dy[t][c];  dH_pre[i] = sum_t sum_c dy[t][c] x[t][i][c] */
/* ------------------------------------------------------------------------ */

int orc_h_aggregate_static_fwd(const double *x, const double *Hpre, int64_t T, int n, int64_t C,
                               double *y)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t)
        for (int64_t c = 0; c < C; ++c) {
            double acc = 0.0;
            for (int i = 0; i < n; ++i) acc += Hpre[i] * x[(t * n + i) * C + c];
            y[t * C + c] = acc;
        }
    return 0;
}

int orc_h_aggregate_static_bwd(const double *dy, const double *x, const double *Hpre, int64_t T,
                               int n, int64_t C, double *dx, double *dHpre)
{
    if (dx) {
#pragma omp parallel for schedule(static)
        for (int64_t t = 0; t < T; ++t)
            for (int i = 0; i < n; ++i)
                for (int64_t c = 0; c < C; ++c) dx[(t * n + i) * C + c] = Hpre[i] * dy[t * C + c];
    }
    if (dHpre) {
#pragma omp parallel for schedule(static)
        for (int i = 0; i < n; ++i) {
            double acc = 0.0;
            for (int64_t t = 0; t < T; ++t)
                for (int64_t c = 0; c < C; ++c) acc += dy[t * C + c] * x[(t * n + i) * C + c];
            dHpre[i] = acc;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* rmsnorm_residual ([rlk] PR body task P1-5 "RMSNorm + residual fork",      */
/* P1-8 "cross-rank dgamma"; the review notes that rmsnorm_residual_fwd      */
/* guards its own zero row; the follow-up commit: the pre-normalization      */
/* intermediate must be exposed).  Reading: the fork h = x + res is both    */
/* returned (the residual that continues) and normalized with a learnable    */
/* per-channel weight gamma:                                                 */
/*   h = x + res;  rho = 1 / sqrt(sum_c h^2 / C + eps);  y = h rho gamma       */
/* res and gamma may be NULL (no residual add; gamma = 1).  Backward, with   */
/* dh the gradient that reaches the fork output h from elsewhere (NULL = 0): */
/*   g = dy gamma;  dx = dres = dh + rho g - rho^3 h (sum_c g h) / C          */
/*   dgamma[c] = sum_t dy[t][c] h[t][c] rho_t   (ascending t)                 */
/* ------------------------------------------------------------------------ */

static double fork_h(const double *x, const double *res, int64_t i)
{
    return res ? x[i] + res[i] : x[i];
}

int orc_rmsnorm_residual_fwd(const double *x, const double *res, const double *gamma,
                             int64_t rows, int64_t cols, double eps, double *h, double *y,
                             double *rstd)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double s = 0.0;
        for (int64_t c = 0; c < cols; ++c) {
            double v = fork_h(x, res, r * cols + c);
            s += v * v;
        }
        double rho = 1.0 / sqrt(s / (double)cols + eps);
        if (rstd) rstd[r] = rho;
        for (int64_t c = 0; c < cols; ++c) {
            double v = fork_h(x, res, r * cols + c);
            if (h) h[r * cols + c] = v;
            if (y) y[r * cols + c] = v * rho * (gamma ? gamma[c] : 1.0);
        }
    }
    return 0;
}

int orc_rmsnorm_residual_bwd(const double *dy, const double *dh, const double *x,
                             const double *res, const double *gamma, int64_t rows, int64_t cols,
                             double eps, double *dx, double *dgamma)
{
    double *rho_all = (double *)malloc(sizeof(double) * (size_t)(rows > 0 ? rows : 1));
    if (!rho_all) return 2;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double s = 0.0, d = 0.0;
        for (int64_t c = 0; c < cols; ++c) {
            double v = fork_h(x, res, r * cols + c);
            s += v * v;
            d += dy[r * cols + c] * (gamma ? gamma[c] : 1.0) * v;
        }
        double rho = 1.0 / sqrt(s / (double)cols + eps);
        rho_all[r] = rho;
        if (dx)
            for (int64_t c = 0; c < cols; ++c) {
                double v = fork_h(x, res, r * cols + c);
                double g = dy[r * cols + c] * (gamma ? gamma[c] : 1.0);
                dx[r * cols + c] = (dh ? dh[r * cols + c] : 0.0) + rho * g -
                                   rho * rho * rho * v * d / (double)cols;
            }
    }
    if (dgamma) {
#pragma omp parallel for schedule(static)
        for (int64_t c = 0; c < cols; ++c) {
            double acc = 0.0;
            for (int64_t r = 0; r < rows; ++r)
                acc += dy[r * cols + c] * fork_h(x, res, r * cols + c) * rho_all[r];
            dgamma[c] = acc;
        }
    }
    free(rho_all);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* proj_rms_compute_h over a channel-sharded residual ([rlk] PR body task    */
/* P1-6 "fp32_gemm_rms TP/SP contract").  Reading: a shard owns channels     */
/* [c0, c1) of every stream, i.e. the K indices k = i*C + c; s = sum x^2 and */
/* u = x.W are sums over K, so a shard computes its partial sums, the        */
/* partials are summed over shards, and compute_h runs on the totals with    */
/* the full K.  In the backward, du and the RMS coefficient are per-token    */
/* values of the totals; each shard forms dx and dW for its own K indices.   */
/* Here a shard's x is [T][n][Cs] and its W rows are k' = i*Cs + c'.          */
/* ------------------------------------------------------------------------ */

int orc_proj_rms_partials(const double *xs, const double *Ws, int64_t T, int n, int64_t Cs,
                          double *u, double *s)
{
    const int O = n * n + 2 * n;
    const int64_t Ks = (int64_t)n * Cs;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double acc[ORC_MAX_N * ORC_MAX_N + 2 * ORC_MAX_N];
        double sq = 0.0;
        for (int o = 0; o < O; ++o) acc[o] = 0.0;
        for (int64_t k = 0; k < Ks; ++k) {
            double xv = xs[t * Ks + k];
            sq += xv * xv;
            for (int o = 0; o < O; ++o) acc[o] += xv * Ws[k * O + o];
        }
        for (int o = 0; o < O; ++o) u[t * O + o] = acc[o];
        s[t] = sq;
    }
    return 0;
}

/* compute_h from the summed partials: q = sqrt(s/K), r = 1/(q + eps_rms),
 * z = alpha_seg r u + b, then the gates and Sinkhorn. */
int orc_compute_h_from_sums(const double *u, const double *s, int64_t K, const double *alpha,
                            const double *b, int64_t T, int n, int iters, double eps_sk,
                            double eps_rms, double *Hpre, double *Hpost, double *Hres,
                            double *r_out)
{
    if (n < 1 || n > ORC_MAX_N) return 1;
    const int O = n * n + 2 * n;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double z[ORC_MAX_N * ORC_MAX_N + 2 * ORC_MAX_N];
        double r = 1.0 / (sqrt(s[t] / (double)K) + eps_rms);
        for (int o = 0; o < O; ++o) z[o] = seg_alpha(alpha, n, o) * r * u[t * O + o] + b[o];
        compute_h_token(z, n, iters, eps_sk, Hpre + t * n, Hpost + t * n, Hres + t * n * n);
        if (r_out) r_out[t] = r;
    }
    return 0;
}

/* Backward of compute_h from the totals: per token du[o] = alpha_seg r dz[o]
 * and coef = dr (-r^2 / (K q)) (0 when q == 0), so that a shard's
 * dx[k] = sum_o du[o] W[k][o] + coef x[k]; dalpha and db as in
 * orc_proj_rms_compute_h_bwd (ascending t).  Any output may be NULL. */
int orc_compute_h_bwd_from_sums(const double *dHpre, const double *dHpost, const double *dHres,
                                const double *u, const double *s, int64_t K,
                                const double *alpha, const double *b, int64_t T, int n,
                                int iters, double eps_sk, double eps_rms, double *du,
                                double *coef, double *dalpha, double *db)
{
    if (n < 1 || n > ORC_MAX_N) return 1;
    const int O = n * n + 2 * n;
    double *ga_all = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * 3);
    double *dz_all = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * O);
    const size_t trace_len = (size_t)(2 * iters + 1) * n * n;
    double *traces = (double *)malloc(sizeof(double) * trace_len * (size_t)(T > 0 ? T : 1));
    if (!ga_all || !dz_all || !traces) {
        free(ga_all); free(dz_all); free(traces);
        return 2;
    }
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        double z[ORC_MAX_N * ORC_MAX_N + 2 * ORC_MAX_N], dz[ORC_MAX_N * ORC_MAX_N + 2 * ORC_MAX_N];
        double g[ORC_MAX_N * ORC_MAX_N];
        const double *ut = u + t * O;
        double q = sqrt(s[t] / (double)K);
        double r = 1.0 / (q + eps_rms);
        for (int o = 0; o < O; ++o) z[o] = seg_alpha(alpha, n, o) * r * ut[o] + b[o];
        for (int i = 0; i < n; ++i) {
            double sp = sigmoid(z[i]);
            double so = sigmoid(z[n + i]);
            dz[i] = dHpre[t * n + i] * sp * (1.0 - sp);
            dz[n + i] = dHpost[t * n + i] * 2.0 * so * (1.0 - so);
        }
        for (int e = 0; e < n * n; ++e) g[e] = dHres[t * n * n + e];
        sinkhorn_bwd_one(g, z + 2 * n, n, iters, eps_sk, dz + 2 * n, traces + (size_t)t * trace_len);
        double ga[3] = {0.0, 0.0, 0.0};
        double dr = 0.0;
        for (int o = 0; o < O; ++o) {
            int sgi = (o < n) ? 0 : (o < 2 * n ? 1 : 2);
            ga[sgi] += dz[o] * r * ut[o];
            dr += dz[o] * seg_alpha(alpha, n, o) * ut[o];
            if (du) du[t * O + o] = seg_alpha(alpha, n, o) * r * dz[o];
            dz_all[t * O + o] = dz[o];
        }
        for (int k = 0; k < 3; ++k) ga_all[t * 3 + k] = ga[k];
        if (coef) coef[t] = (q > 0.0) ? dr * (-(r * r) / ((double)K * q)) : 0.0;
    }
    if (dalpha) {
        for (int k = 0; k < 3; ++k) dalpha[k] = 0.0;
        for (int64_t t = 0; t < T; ++t)
            for (int k = 0; k < 3; ++k) dalpha[k] += ga_all[t * 3 + k];
    }
    if (db) {
        for (int o = 0; o < O; ++o) db[o] = 0.0;
        for (int64_t t = 0; t < T; ++t)
            for (int o = 0; o < O; ++o) db[o] += dz_all[t * O + o];
    }
    free(ga_all); free(dz_all); free(traces);
    return 0;
}

/* A shard's part of the projection backward:
 *   dx[t][k'] = sum_o du[t][o] W[k'][o] + coef[t] x[t][k'];  dW[k'][o] = sum_t x[t][k'] du[t][o] */
int orc_proj_rms_partial_bwd(const double *xs, const double *Ws, const double *du,
                             const double *coef, int64_t T, int n, int64_t Cs, double *dx,
                             double *dW)
{
    const int O = n * n + 2 * n;
    const int64_t Ks = (int64_t)n * Cs;
    if (dx) {
#pragma omp parallel for schedule(static)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t k = 0; k < Ks; ++k) {
                double acc = 0.0;
                for (int o = 0; o < O; ++o) acc += du[t * O + o] * Ws[k * O + o];
                dx[t * Ks + k] = acc + coef[t] * xs[t * Ks + k];
            }
    }
    if (dW) {
#pragma omp parallel for schedule(static)
        for (int64_t k = 0; k < Ks; ++k)
            for (int o = 0; o < O; ++o) {
                double acc = 0.0;
                for (int64_t t = 0; t < T; ++t) acc += xs[t * Ks + k] * du[t * O + o];
                dW[k * O + o] = acc;
            }
    }
    return 0;
}

int orc_num_threads(void)
{
    int nt = 1;
#ifdef _OPENMP
#pragma omp parallel
    {
#pragma omp single
        nt = omp_get_num_threads();
    }
#endif
    return nt;
}
