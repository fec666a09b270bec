/*
 * libmhc: mHC (Manifold-Constrained Hyper-Connections) residual-stream ops
 * for NVIDIA GB300 (sm_103a), forward and backward, behind a plain C ABI.
 *
 * Sources for the operations (web pages):
 *  [rwkv]  rwkv-ops 0.6.1, rwkv_ops/mhc_kernel/jax_kernel/mhu_ffi.cu: the
 *          XLA-FFI handlers SinkhornFwdHost/SinkhornBwdHost, RMSNormFwdHost/
 *          RMSNormBwdHost, StreamAggregateFwd/Bwd, MhcPostOpFwdHost/
 *          MhcPostOpBwdHost, MhcPreOpFwdHost/MhcPreOpBwdHost.
 *  [mcore] Megatron-Core API docs, core.fusions.fused_mhc_kernels: the four
 *          fused ops fused_sinkhorn, fused_h_aggregate, fused_h_post_bda,
 *          fused_proj_rms_compute_h, and the torch backward helpers
 *          _torch_h_aggregate_bwd, _torch_h_post_bda_bwd.
 *  [rlk]   RL-Align/RL-Kernel PR #383 (P1 start kit, mHC + RMSNorm): the
 *          fp32_gemm_rms forward/backward (RMS r = 1/(q + eps), zero-row
 *          guard) and the three alpha scalars over PRE/POST/COMB.
 *
 * Notation.  T tokens, n streams (4 or 8), C hidden size, K = n*C,
 * O = n*n + 2*n controller logits.  The residual x is [T, n, C] bf16
 * (row-major; flattened index k = i*C + c).  W is [K, O] fp32 row-major.
 * alpha3 = (alpha_pre, alpha_post, alpha_res).  b is [O] fp32.  Logit order
 * is pre[0,n) | post[n,2n) | res[2n, 2n+n*n), res row-major.  H_pre, H_post
 * are [T, n] fp32; H_res is [T, n, n] fp32 and H_res[t][j][i] carries
 * residual stream j into output stream i.
 *
 * Conventions (every entry point):
 *  - Pointers are DEVICE pointers owned by the caller.  The library
 *    allocates no device memory; ops that need scratch take (ws, ws_bytes)
 *    sized by mhc_workspace_bytes().  ws must be 256-byte aligned.
 *  - All work is enqueued on `stream`; calls return before it completes.
 *  - Every output is fully overwritten; nothing needs zeroing first.
 *  - Arguments are validated on the host before any launch.  A failed check
 *    returns a nonzero mhc_status, launches nothing and writes nothing;
 *    mhc_last_error() then describes it (thread-local).
 *  - Every pointer must be 16-byte aligned and C a multiple of 8.  n must be
 *    4 or 8; 0 <= iters <= 64.  The ops that take W (they run on the tensor
 *    cores with 32-bit TMA coordinates) need T < 2^31 and n*C < 2^31.
 *  - T (or M, rows) may be 0: the call then returns MHC_OK and does nothing.
 *  - Results are deterministic: no atomics, fixed reduction order; the same
 *    inputs give bitwise identical outputs run to run.
 *  - A kernel that detects an internal fault (a bounded wait that timed
 *    out) sets a device-side error word and returns early;
 *    mhc_device_error() reads and clears it.
 */
#ifndef MHC_H_
#define MHC_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MHC_API __attribute__((visibility("default")))
#else
#define MHC_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* bf16 values are passed as their 16-bit storage. */
typedef uint16_t mhc_bf16;
/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *mhc_stream_t;

typedef enum {
    MHC_OK = 0,
    MHC_ERR_NULL_PTR = 1,            /* a required pointer is NULL */
    MHC_ERR_BAD_SHAPE = 2,           /* negative size, C % 8 != 0, overflow */
    MHC_ERR_MISALIGNED = 3,          /* pointer alignment rule broken */
    MHC_ERR_UNSUPPORTED_N = 4,       /* n not in {4, 8} */
    MHC_ERR_WORKSPACE_TOO_SMALL = 5, /* ws_bytes < mhc_workspace_bytes() */
    MHC_ERR_BAD_ARG = 6,             /* iters out of range, eps < 0 or NaN */
    MHC_ERR_CUDA = 7,                /* a CUDA runtime call failed */
    MHC_ERR_NO_DEVICE = 8,           /* no usable sm_103 device */
    MHC_ERR_DEVICE_FAULT = 9         /* a kernel reported an internal fault */
} mhc_status;

#define MHC_MAX_ITERS 64

/* Text for a status code (static storage). */
MHC_API const char *mhc_status_string(mhc_status s);
/* Message of the last failing call on this host thread ("" if none). */
MHC_API const char *mhc_last_error(void);
/* Library version, major*10000 + minor*100 + patch. */
MHC_API int mhc_version(void);

/* Batch-invariant mode ([rlk] PR body: the fixed-K / batch-invariant GEMM
 * reference of task P1-2).  Off by default.  When on, the forward
 * projection's K splits are a function of K alone (4096-wide), so every
 * per-token output of every op (H_*, u, r, y, out, dx, df, ...) is bitwise
 * independent of T and of the token's position in the batch; the sums over
 * tokens (dW, dalpha, db, dbias, dgamma) are deterministic for a given T.
 * Process-wide; workspace sizes depend on it, so query them after setting
 * it, and do not change it while calls are in flight. */
MHC_API void mhc_set_batch_invariant(int on);
MHC_API int mhc_batch_invariant(void);

/* Bit-reproducible mode (RL-Align/RL-Kernel PR #383, PR body, "Numerical
 * contract": fp32 arithmetic and only two reduction trees, a serial
 * ascending left fold for long reductions and (a0 + a1) + (a2 + a3) over the
 * four streams).  When on, mhc_sinkhorn_fwd/bwd, mhc_proj_rms_compute_h_fwd/
 * bwd, mhc_h_aggregate_fwd/bwd, mhc_h_post_bda_fwd/bwd and mhc_layer_fwd/bwd
 * compute every result in that order: each stream sum is the four-stream
 * tree, each sum over channels, over K, over the controller logits or over
 * tokens (dH_*, u, sum x^2, dx_proj, dW, dalpha, db, dbias) is a serial fold
 * in ascending index order, every product is rounded before it is added, and
 * exp is the library's own (Cody-Waite reduction, Taylor polynomial), so the
 * results are the same bits on every device and in any program that
 * performs those fp32 operations in that order.  Defined for n = 4: with the
 * mode on these calls return MHC_ERR_UNSUPPORTED_N for n = 8.  The mode uses
 * plain (slow) kernels; the backward recomputes u, r from x and ignores
 * u_save, r_save.  Process-wide; do not change it while calls are in flight.
 * The other entry points (RMSNorm, the next-row ops) are not affected. */
MHC_API void mhc_set_pinned_reductions(int on);
MHC_API int mhc_pinned_reductions(void);

/* Synchronises `stream`, reads and clears the device-side fault word.
 * Returns MHC_OK if no kernel reported a fault, MHC_ERR_DEVICE_FAULT
 * otherwise (*code receives the fault code, 0 if none; code may be NULL). */
MHC_API mhc_status mhc_device_error(int *code, mhc_stream_t stream);

/* Self-test of that path: launches one kernel whose bounded wait, the same
 * wait the tensor-core kernels use, is on an mbarrier that nothing arrives
 * at; after about wait_us microseconds of SM clock (1 <= wait_us <= 1e6) it
 * gives up, records fault code 105 in the device error word and returns.
 * Nothing faults or hangs, and the context stays usable; a following
 * mhc_device_error() returns MHC_ERR_DEVICE_FAULT with code 105. */
MHC_API mhc_status mhc_selftest_wait_timeout(int wait_us, mhc_stream_t stream);

typedef enum {
    MHC_OP_PROJ_RMS_COMPUTE_H_FWD = 1,
    MHC_OP_PROJ_RMS_COMPUTE_H_BWD = 2,
    MHC_OP_H_POST_BDA_BWD = 3,
    MHC_OP_LAYER_FWD = 4,
    MHC_OP_LAYER_BWD = 5,
    MHC_OP_RMSNORM_RESIDUAL_BWD = 6,   /* (rows, -, cols); only when dgamma is wanted */
    MHC_OP_H_AGGREGATE_RMSNORM_BWD = 7, /* only when dgamma is wanted */
    MHC_OP_H_AGGREGATE_STATIC_BWD = 8,
    MHC_OP_PROJ_RMS_PARTIAL_FWD = 9,   /* C = the shard's channels Cs */
    MHC_OP_COMPUTE_H_BWD = 10,
    MHC_OP_PROJ_RMS_PARTIAL_BWD = 11,  /* C = the shard's channels Cs */
    MHC_OP_H_POST_BDA_COMPUTE_H_FWD = 12
} mhc_op;

/* Workspace bytes an op needs for (T, n, C); 0 for a bad op or shape.
 * The other ops need none.  MHC_OP_RMSNORM_RESIDUAL_BWD ignores n. */
MHC_API size_t mhc_workspace_bytes(mhc_op op, int64_t T, int n, int64_t C);

/* ------------------------------------------------------------------ */
/* Sinkhorn-Knopp, batched ([rwkv] SinkhornFwdHost/SinkhornBwdHost,    */
/* [mcore] fused_sinkhorn).                                            */
/* ------------------------------------------------------------------ */

/* P = Sinkhorn(exp(logits)) for M independent n x n matrices.
 * logits, P: [M, n, n] fp32.  A = exp(logits); then `iters` times every row
 * of A is divided by (its sum + eps) and then every column by (its sum +
 * eps).  One launch for the whole batch. */
MHC_API mhc_status mhc_sinkhorn_fwd(const float *logits, float *P, int64_t M, int n, int iters,
                            float eps, mhc_stream_t stream);

/* dlogits = gradient of sum(dP * P) through the unrolled iteration above.
 * dP, logits, dlogits: [M, n, n] fp32.  The forward is recomputed. */
MHC_API mhc_status mhc_sinkhorn_bwd(const float *dP, const float *logits, float *dlogits, int64_t M,
                            int n, int iters, float eps, mhc_stream_t stream);

/* ------------------------------------------------------------------ */
/* proj_rms_compute_h ([mcore] fused_proj_rms_compute_h; [rlk]         */
/* fp32_gemm_rms; [rwkv] MhcPreOpFwdHost output gates).                */
/* ------------------------------------------------------------------ */

/* Per token t:
 *   s = sum_k x[t][k]^2,  q = sqrt(s/K),  r = 1/(q + eps_rms)
 *   u[o] = sum_k x[t][k] W[k][o]                        (fp32 result)
 *   z[o] = alpha_seg(o) * r * u[o] + b[o]
 *   H_pre = sigmoid(z_pre), H_post = 2 sigmoid(z_post),
 *   H_res = Sinkhorn(exp(z_res)) as mhc_sinkhorn_fwd with eps_sk.
 * Outputs H_pre [T,n], H_post [T,n], H_res [T,n,n]; u_save [T,O] and
 * r_save [T] (both may be NULL) keep u and r for the backward.
 * ws: mhc_workspace_bytes(MHC_OP_PROJ_RMS_COMPUTE_H_FWD, T, n, C). */
MHC_API mhc_status mhc_proj_rms_compute_h_fwd(const mhc_bf16 *x, const float *W, const float *alpha3,
                                      const float *b, int64_t T, int n, int64_t C, int iters,
                                      float eps_sk, float eps_rms, float *H_pre, float *H_post,
                                      float *H_res, float *u_save, float *r_save, void *ws,
                                      size_t ws_bytes, mhc_stream_t stream);

/* Backward of the above for upstream grads dH_pre [T,n], dH_post [T,n],
 * dH_res [T,n,n] (fp32).  u_save and r_save (required) come from the
 * forward.  Per token:
 *   dz_pre = dH_pre s(1-s), dz_post = 2 dH_post s(1-s) (s the gate's sigmoid),
 *   dz_res = Sinkhorn backward of dH_res,
 *   du = alpha_seg r dz,  dr = sum_o dz alpha_seg u,
 *   dx[t][k] = sum_o du[o] W[k][o] - dr r^2 x[t][k] / (K q)  (last term 0
 *   when q == 0, an all-zero row).
 * Outputs dx [T,n,C] bf16, dW [K,O] = sum_t x^T du, dalpha3 [3] =
 * sum over tokens and segment of dz r u, db [O] = sum_t dz (all fp32).
 * ws: mhc_workspace_bytes(MHC_OP_PROJ_RMS_COMPUTE_H_BWD, T, n, C). */
MHC_API mhc_status mhc_proj_rms_compute_h_bwd(const float *dH_pre, const float *dH_post,
                                      const float *dH_res, const mhc_bf16 *x, const float *W,
                                      const float *alpha3, const float *b, const float *u_save,
                                      const float *r_save, int64_t T, int n, int64_t C,
                                      int iters, float eps_sk, float eps_rms, mhc_bf16 *dx,
                                      float *dW, float *dalpha3, float *db, void *ws,
                                      size_t ws_bytes, mhc_stream_t stream);

/* ------------------------------------------------------------------ */
/* h_aggregate ([mcore] fused_h_aggregate / FusedHAggregate,           */
/* _torch_h_aggregate_bwd; [rwkv] StreamAggregateFwd/Bwd).             */
/* ------------------------------------------------------------------ */

/* y[t][c] = sum_i H_pre[t][i] x[t][i][c].  x [T,n,C] bf16, H_pre [T,n] fp32,
 * y [T,C] bf16 (one rounding of the fp32 sum). */
MHC_API mhc_status mhc_h_aggregate_fwd(const mhc_bf16 *x, const float *H_pre, mhc_bf16 *y, int64_t T,
                               int n, int64_t C, mhc_stream_t stream);

/* dx[t][i][c] = H_pre[t][i] dy[t][c] (bf16), dH_pre[t][i] = sum_c dy x (fp32). */
MHC_API mhc_status mhc_h_aggregate_bwd(const mhc_bf16 *dy, const mhc_bf16 *x, const float *H_pre,
                               mhc_bf16 *dx, float *dH_pre, int64_t T, int n, int64_t C,
                               mhc_stream_t stream);

/* ------------------------------------------------------------------ */
/* h_post_bda ([mcore] fused_h_post_bda "H_res.T @ residual + H_post * */
/* (x + bias)", _torch_h_post_bda_bwd; [rwkv] MhcPostOpFwd/BwdHost).   */
/* Dropout is not applied (p = 0).                                     */
/* ------------------------------------------------------------------ */

/* out[t][i][c] = sum_j H_res[t][j][i] residual[t][j][c]
 *               + H_post[t][i] (f[t][c] + bias[c])
 * residual, out [T,n,C] bf16; f [T,C] bf16; bias [C] bf16 or NULL (zero). */
MHC_API mhc_status mhc_h_post_bda_fwd(const mhc_bf16 *residual, const mhc_bf16 *f, const mhc_bf16 *bias,
                              const float *H_res, const float *H_post, mhc_bf16 *out, int64_t T,
                              int n, int64_t C, mhc_stream_t stream);

/* dresidual[t][j][c] = sum_i H_res[t][j][i] dout[t][i][c]       (bf16)
 * df[t][c]           = sum_i H_post[t][i] dout[t][i][c]          (bf16)
 * dbias[c]           = sum_t df[t][c] (from fp32 df; NULL to skip)
 * dH_res[t][j][i]    = sum_c residual[t][j][c] dout[t][i][c]     (fp32)
 * dH_post[t][i]      = sum_c dout[t][i][c] (f[t][c] + bias[c])   (fp32)
 * ws: mhc_workspace_bytes(MHC_OP_H_POST_BDA_BWD, T, n, C). */
MHC_API mhc_status mhc_h_post_bda_bwd(const mhc_bf16 *dout, const mhc_bf16 *residual, const mhc_bf16 *f,
                              const mhc_bf16 *bias, const float *H_res, const float *H_post,
                              mhc_bf16 *dresidual, mhc_bf16 *df, float *dbias, float *dH_res,
                              float *dH_post, int64_t T, int n, int64_t C, void *ws,
                              size_t ws_bytes, mhc_stream_t stream);

/* ------------------------------------------------------------------ */
/* Standalone RMSNorm, no weight ([rwkv] RMSNormFwdHost/BwdHost).       */
/* ------------------------------------------------------------------ */

/* rho = 1/sqrt(mean_c x^2 + eps); y = x rho.  x, y [rows, cols] bf16;
 * rstd [rows] fp32 receives rho (may be NULL).  cols % 8 == 0. */
MHC_API mhc_status rmsnorm_fwd(const mhc_bf16 *x, mhc_bf16 *y, float *rstd, int64_t rows, int64_t cols,
                       float eps, mhc_stream_t stream);

/* dx = rho dy - rho^3 x (sum_c dy x) / cols.  rstd from the forward, or NULL
 * to recompute rho from x. */
MHC_API mhc_status rmsnorm_bwd(const mhc_bf16 *dy, const mhc_bf16 *x, const float *rstd, mhc_bf16 *dx,
                       int64_t rows, int64_t cols, float eps, mhc_stream_t stream);

/* ------------------------------------------------------------------ */
/* h_aggregate with one static H_pre [n] for every token ([rwkv]        */
/* StreamAggregateFwd/Bwd with per_token = false: H_pre [n], d_H_pre [n]).*/
/* ------------------------------------------------------------------ */

/* y[t][c] = sum_i H_pre[i] x[t][i][c].  x [T,n,C] bf16, H_pre [n] fp32,
 * y [T,C] bf16. */
MHC_API mhc_status mhc_h_aggregate_static_fwd(const mhc_bf16 *x, const float *H_pre, mhc_bf16 *y,
                                              int64_t T, int n, int64_t C, mhc_stream_t stream);

/* dx[t][i][c] = H_pre[i] dy[t][c] (bf16; dx may be NULL),
 * dH_pre[i] = sum_t sum_c dy[t][c] x[t][i][c] (fp32 [n], fixed summation order).
 * ws: mhc_workspace_bytes(MHC_OP_H_AGGREGATE_STATIC_BWD, T, n, C).  T = 0
 * writes dH_pre = 0. */
MHC_API mhc_status mhc_h_aggregate_static_bwd(const mhc_bf16 *dy, const mhc_bf16 *x,
                                              const float *H_pre, mhc_bf16 *dx, float *dH_pre,
                                              int64_t T, int n, int64_t C, void *ws,
                                              size_t ws_bytes, mhc_stream_t stream);

/* ------------------------------------------------------------------ */
/* rmsnorm_residual: RMSNorm with a residual fork and a learnable       */
/* weight ([rlk] PR body tasks P1-5 "RMSNorm + residual fork" and P1-8  */
/* "cross-rank dgamma"; the follow-up commit: the pre-normalization     */
/* intermediate is exposed).                                           */
/* ------------------------------------------------------------------ */

/* h = x + res (res NULL: h = x), rho = 1/sqrt(mean_c h^2 + eps),
 * y = h rho gamma (gamma NULL: 1).  x, res, h, y [rows, cols] bf16; gamma
 * [cols] fp32; rstd [rows] fp32.  h (the fork) and rstd may be NULL.  The
 * norm uses the fp32 sum; h is its bf16 rounding.  cols % 8 == 0,
 * cols <= 32768. */
MHC_API mhc_status rmsnorm_residual_fwd(const mhc_bf16 *x, const mhc_bf16 *res,
                                        const float *gamma, mhc_bf16 *h, mhc_bf16 *y,
                                        float *rstd, int64_t rows, int64_t cols, float eps,
                                        mhc_stream_t stream);

/* With g = dy gamma:
 *   dx = dres = dh + rho g - rho^3 h (sum_c g h) / cols     (bf16; the one
 *        gradient of both x and res; dh, the gradient reaching the fork
 *        output h from elsewhere, may be NULL = 0)
 *   dgamma[c] = sum_t dy h rho (fp32 [cols], fixed order; NULL to skip).
 * rstd from the forward, or NULL to recompute rho.
 * ws: mhc_workspace_bytes(MHC_OP_RMSNORM_RESIDUAL_BWD, rows, 0, cols), needed
 * only with dgamma.  rows = 0 writes dgamma = 0. */
MHC_API mhc_status rmsnorm_residual_bwd(const mhc_bf16 *dy, const mhc_bf16 *dh,
                                        const mhc_bf16 *x, const mhc_bf16 *res,
                                        const float *gamma, const float *rstd, mhc_bf16 *dx,
                                        float *dgamma, int64_t rows, int64_t cols, float eps,
                                        void *ws, size_t ws_bytes, mhc_stream_t stream);

/* ------------------------------------------------------------------ */
/* h_aggregate followed by the weighted RMSNorm of its output, in one   */
/* pass over x ([mcore] fused_h_aggregate; [rlk] rmsnorm_residual).     */
/* ------------------------------------------------------------------ */

/* y = sum_i H_pre[t][i] x_i (the pre-normalization intermediate; bf16 [T,C],
 * may be NULL), yn = y rho gamma with rho = 1/sqrt(mean_c y^2 + eps) from
 * the fp32 y (bf16 [T,C]); rstd [T] fp32 (may be NULL).  H_pre [T,n] fp32,
 * gamma [C] fp32 or NULL.  C <= 32768. */
MHC_API mhc_status mhc_h_aggregate_rmsnorm_fwd(const mhc_bf16 *x, const float *H_pre,
                                               const float *gamma, mhc_bf16 *y, mhc_bf16 *yn,
                                               float *rstd, int64_t T, int n, int64_t C,
                                               float eps, mhc_stream_t stream);

/* With dy_total = dy + rho g - rho^3 y (sum_c g y)/C, g = dyn gamma (dy, the
 * gradient reaching y from elsewhere, may be NULL):
 *   dx[t][i][c] = H_pre[t][i] dy_total (bf16), dH_pre[t][i] = sum_c dy_total x_i
 *   (fp32), dgamma[c] = sum_t dyn y rho (fp32, fixed order; NULL to skip).
 * rstd from the forward or NULL to recompute.  ws:
 * mhc_workspace_bytes(MHC_OP_H_AGGREGATE_RMSNORM_BWD, T, n, C), only with dgamma. */
MHC_API mhc_status mhc_h_aggregate_rmsnorm_bwd(const mhc_bf16 *dyn, const mhc_bf16 *dy,
                                               const mhc_bf16 *x, const float *H_pre,
                                               const float *gamma, const float *rstd,
                                               mhc_bf16 *dx, float *dH_pre, float *dgamma,
                                               int64_t T, int n, int64_t C, float eps, void *ws,
                                               size_t ws_bytes, mhc_stream_t stream);

/* ------------------------------------------------------------------ */
/* proj_rms_compute_h over channel shards ([rlk] PR body task P1-6,     */
/* the fp32_gemm_rms TP/SP contract).  A shard owns channels [c0, c1)  */
/* of every stream: x_shard [T, n, Cs] bf16 and W_shard [n*Cs, O] fp32 */
/* with rows i*Cs + c' (the rows i*C + c0 + c' of W).  Each shard      */
/* computes partial sums; the caller sums them over shards (an         */
/* all-reduce); compute_h runs on the totals with the full K = n*C;    */
/* each shard forms dx and dW for its own channels from the per-token  */
/* du and RMS coefficient.                                             */
/* ------------------------------------------------------------------ */

/* u_part[t][o] = sum_{k in shard} x[t][k] W[k][o], s_part[t] = sum_{k in shard} x^2
 * (fp32).  ws: mhc_workspace_bytes(MHC_OP_PROJ_RMS_PARTIAL_FWD, T, n, Cs). */
MHC_API mhc_status mhc_proj_rms_partial_fwd(const mhc_bf16 *x_shard, const float *W_shard,
                                            int64_t T, int n, int64_t Cs, float *u_part,
                                            float *s_part, void *ws, size_t ws_bytes,
                                            mhc_stream_t stream);

/* compute_h from the totals u [T,O], s [T]: r = 1/(sqrt(s/K) + eps_rms),
 * z = alpha_seg r u + b, gates and Sinkhorn as mhc_proj_rms_compute_h_fwd.
 * r_save [T] may be NULL. */
MHC_API mhc_status mhc_compute_h_fwd(const float *u, const float *s, int64_t K,
                                     const float *alpha3, const float *b, int64_t T, int n,
                                     int iters, float eps_sk, float eps_rms, float *H_pre,
                                     float *H_post, float *H_res, float *r_save,
                                     mhc_stream_t stream);

/* Per-token backward coefficients from the totals: du[t][o] = alpha_seg r dz[o]
 * ([T,O] fp32) and coef[t] = -dr r^2/(K q) ([T]; 0 for an all-zero row), so
 * that a shard's dx = du W_shard^T + coef x_shard; dalpha3 [3], db [O] summed
 * over tokens (fixed order).  ws: mhc_workspace_bytes(MHC_OP_COMPUTE_H_BWD, T, n, 8). */
MHC_API mhc_status mhc_compute_h_bwd(const float *dH_pre, const float *dH_post,
                                     const float *dH_res, const float *u, const float *s,
                                     int64_t K, const float *alpha3, const float *b, int64_t T,
                                     int n, int iters, float eps_sk, float eps_rms, float *du,
                                     float *coef, float *dalpha3, float *db, void *ws,
                                     size_t ws_bytes, mhc_stream_t stream);

/* A shard's dx_shard[t][k'] = sum_o du[t][o] W_shard[k'][o] + coef[t] x_shard[t][k']
 * (bf16) and dW_shard[k'][o] = sum_t x_shard[t][k'] du[t][o] (fp32).
 * ws: mhc_workspace_bytes(MHC_OP_PROJ_RMS_PARTIAL_BWD, T, n, Cs). */
MHC_API mhc_status mhc_proj_rms_partial_bwd(const mhc_bf16 *x_shard, const float *W_shard,
                                            const float *du, const float *coef, int64_t T,
                                            int n, int64_t Cs, mhc_bf16 *dx_shard,
                                            float *dW_shard, void *ws, size_t ws_bytes,
                                            mhc_stream_t stream);

/* ------------------------------------------------------------------ */
/* Cross-layer fusion: the h_post_bda of layer l, whose output is the   */
/* residual input of layer l+1, with the proj_rms_compute_h forward of  */
/* layer l+1 on it ([rlk] PR body: fusing fp32_gemm_rms with the op     */
/* that produces its input; [mcore] fused_h_post_bda followed by         */
/* fused_proj_rms_compute_h).  The projection pass then reads no HBM of  */
/* its own: out is summed and projected while it is written.            */
/* ------------------------------------------------------------------ */

/* out[t][i][c] = sum_j H_res[t][j][i] residual[t][j][c] + H_post[t][i] (f[t][c] + bias[c])
 * exactly as mhc_h_post_bda_fwd (bf16, bitwise the same), and on x' = out as
 * stored: H_pre_next, H_post_next, H_res_next (and the saves u_save_next
 * [T,O], r_save_next [T], both nullable) exactly as mhc_proj_rms_compute_h_fwd
 * with W_next [K,O], alpha3_next, b_next (the same values up to the order of
 * the fp32 sums over K).  Shapes, alignment and bias as the two ops.
 * ws: mhc_workspace_bytes(MHC_OP_H_POST_BDA_COMPUTE_H_FWD, T, n, C). */
MHC_API mhc_status mhc_h_post_bda_compute_h_fwd(
    const mhc_bf16 *residual, const mhc_bf16 *f, const mhc_bf16 *bias, const float *H_res,
    const float *H_post, const float *W_next, const float *alpha3_next, const float *b_next,
    int64_t T, int n, int64_t C, int iters, float eps_sk, float eps_rms, mhc_bf16 *out,
    float *H_pre_next, float *H_post_next, float *H_res_next, float *u_save_next,
    float *r_save_next, void *ws, size_t ws_bytes, mhc_stream_t stream);

/* ------------------------------------------------------------------ */
/* Per-kernel timing (off by default).  When enabled, every kernel the  */
/* library launches is bracketed by CUDA events on its stream.          */
/* ------------------------------------------------------------------ */

typedef struct {
    char name[48];    /* kernel name */
    int64_t launches; /* launches since the last collect */
    double total_ms;  /* summed event-measured duration */
} mhc_kernel_time;

/* Switch event recording on (nonzero) or off.  Not an error without a GPU. */
MHC_API void mhc_profiler_enable(int on);
/* Waits for the recorded events, writes up to `max` per-kernel totals to
 * `out` (may be NULL), forgets the records and returns the number of
 * distinct kernels seen. */
MHC_API int mhc_profiler_collect(mhc_kernel_time *out, int max);

/* ------------------------------------------------------------------ */
/* One mHC layer (the measured unit): forward proj_rms_compute_h ->     */
/* h_aggregate -> h_post_bda with the sub-layer output f given; backward */
/* the three op backwards and the three-way residual-gradient sum       */
/* ([mcore] fused_add_3), fused into three passes over HBM.             */
/* ------------------------------------------------------------------ */

/* Outputs H_pre, H_post, H_res, u_save, r_save (as the op above; all
 * required), y [T,C] and out [T,n,C] (bf16).
 * ws: mhc_workspace_bytes(MHC_OP_LAYER_FWD, T, n, C). */
MHC_API mhc_status mhc_layer_fwd(const mhc_bf16 *x, const float *W, const float *alpha3, const float *b,
                         const mhc_bf16 *f, const mhc_bf16 *bias, int64_t T, int n, int64_t C,
                         int iters, float eps_sk, float eps_rms, float *H_pre, float *H_post,
                         float *H_res, float *u_save, float *r_save, mhc_bf16 *y,
                         mhc_bf16 *out, void *ws, size_t ws_bytes, mhc_stream_t stream);

/* Gradients of L = <dout, out> + <dy, y> given the forward's saves:
 * dx [T,n,C] bf16 (= d_residual + d_aggregate + d_projection),
 * df [T,C] bf16, dW [K,O], dalpha3 [3], db [O], dbias [C] (fp32; dbias may
 * be NULL when bias is NULL).
 * ws: mhc_workspace_bytes(MHC_OP_LAYER_BWD, T, n, C). */
MHC_API mhc_status mhc_layer_bwd(const mhc_bf16 *dout, const mhc_bf16 *dy, const mhc_bf16 *x,
                         const float *W, const float *alpha3, const float *b, const mhc_bf16 *f,
                         const mhc_bf16 *bias, const float *H_pre, const float *H_post,
                         const float *H_res, const float *u_save, const float *r_save,
                         int64_t T, int n, int64_t C, int iters, float eps_sk, float eps_rms,
                         mhc_bf16 *dx, mhc_bf16 *df, float *dW, float *dalpha3, float *db,
                         float *dbias, void *ws, size_t ws_bytes, mhc_stream_t stream);

/* ------------------------------------------------------------------ */
/* Allocation-free variant.  The web pages have no counterpart of this  */
/* entry point; it exists for callers that cannot allocate device       */
/* memory for a workspace: allocator-free runtimes, plugins that may    */
/* not own device memory, paths that must not call cudaMalloc/cudaFree  */
/* (they can synchronise the device).                                   */
/* ------------------------------------------------------------------ */

/* Size of the fixed scratch array the variant below uses (8 MiB).  It is
 * device global memory inside the library image, held on every GPU that
 * loads the library until the process exits. */
#define MHC_NOALLOC_SCRATCH_BYTES (((size_t)8) << 20)

/* mhc_proj_rms_compute_h_fwd without a workspace argument: the same
 * computation and outputs, with the scratch taken from the library's fixed
 * array.  Calls that would need more scratch than MHC_NOALLOC_SCRATCH_BYTES
 * (mhc_workspace_bytes(MHC_OP_PROJ_RMS_COMPUTE_H_FWD, T, n, C)) return
 * MHC_ERR_WORKSPACE_TOO_SMALL without launching anything.  The size needed
 * grows with T and C and depends on mhc_set_batch_invariant (which fixes the
 * number of K splits): T = 16384, n = 4, C = 4096 needs about 5.9 MB by
 * default, 8.75 MB (rejected) in batch-invariant mode; at n = 8 only small
 * T and C fit (the split copy of W takes 3840 * C bytes, the partial sums up
 * to 32 * T * 320 bytes).  Allocates no memory.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) for that device and caches it; make it before any
 * stream capture.  The cached address belongs to the context current at
 * that first call (the primary context, for CUDA-runtime users) and is not
 * valid after cudaDeviceReset.  All calls share the one array: calls that
 * overlap on the GPU race on it and must be ordered by the caller (same
 * stream, or events). */
MHC_API mhc_status mhc_proj_rms_compute_h_fwd_noalloc(const mhc_bf16 *x, const float *W,
                                                      const float *alpha3, const float *b,
                                                      int64_t T, int n, int64_t C, int iters,
                                                      float eps_sk, float eps_rms,
                                                      float *H_pre, float *H_post,
                                                      float *H_res, float *u_save,
                                                      float *r_save, mhc_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MHC_H_ */
