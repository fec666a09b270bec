// Host-side launchers of the mHC kernels (C++ linkage, internal to libmhc).
// Arguments are already validated by the C-ABI layer in abi.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "common.cuh"

namespace mhc {

typedef __nv_bfloat16 bf16;

// Workspace carving: every sub-buffer starts on a 256-byte boundary.
inline size_t ws_align(size_t b) { return (b + 255) & ~size_t(255); }

constexpr int kMaxIters = 64;
// Split counts of the split reductions are chosen for this many SMs on every
// device, so that results do not depend on the device's SM count.
constexpr int kSplitSms = 152;

int num_sms();

// Raises a kernel's dynamic shared-memory limit to `bytes`, once per device
// and kernel (k_stream.cu).  The attribute call is not stream-ordered, so after
// the first call of each op nothing but launches reaches the stream (the
// calls can be captured into a CUDA graph).
cudaError_t set_smem_limit(const void *kernel, int bytes);

// Sets the thread-local text that mhc_last_error() returns (abi.cu).
void set_error_message(const char *msg);

// Per-kernel event timing (prof.cu); a no-op unless mhc_profiler_enable(1).
void prof_begin(const char *name, cudaStream_t s);
void prof_end(cudaStream_t s);
struct ProfScope {
    cudaStream_t s_;
    ProfScope(const char *name, cudaStream_t s) : s_(s) { prof_begin(name, s); }
    ~ProfScope() { prof_end(s_); }
};
#define MHC_PROF_CAT2(a, b) a##b
#define MHC_PROF_CAT(a, b) MHC_PROF_CAT2(a, b)
// Time the launch(es) in the rest of the enclosing scope under `name`.
#define MHC_PROF(name, s) ::mhc::ProfScope MHC_PROF_CAT(prof_scope_, __LINE__)(name, s)

// Launches `kernel` on stream s with programmatic stream serialization
// allowed: the grid may start its setup while the previous kernel drains,
// and waits in pdl_wait() for that kernel's completion before any memory
// access.
template <class... KArgs, class... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t s, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// k_sinkhorn.cu
cudaError_t launch_sinkhorn_fwd(const float *logits, float *P, int64_t M, int n, int iters,
                                float eps, cudaStream_t s);
cudaError_t launch_sinkhorn_bwd(const float *dP, const float *logits, float *dlogits, int64_t M,
                                int n, int iters, float eps, cudaStream_t s);

// k_stream.cu
// per_token: H_pre is [T][n]; else one static H_pre [n] for every token.
cudaError_t launch_aggregate_fwd(const bf16 *x, const float *Hpre, bf16 *y, int64_t T, int n,
                                 int64_t C, cudaStream_t s, bool per_token = true);
// Static-H_pre backward: dH_pre [n] summed over tokens; scratch agg_static_ws_bytes.
size_t agg_static_ws_bytes(int64_t T, int n);
cudaError_t launch_aggregate_bwd_static(const bf16 *dy, const bf16 *x, const float *Hpre,
                                        bf16 *dx, float *dHpre, int64_t T, int n, int64_t C,
                                        void *ws, cudaStream_t s);
cudaError_t launch_aggregate_bwd(const bf16 *dy, const bf16 *x, const float *Hpre, bf16 *dx,
                                 float *dHpre, int64_t T, int n, int64_t C, cudaStream_t s);
cudaError_t launch_post_fwd(const bf16 *res, const bf16 *f, const bf16 *bias, const float *Hres,
                            const float *Hpost, bf16 *out, int64_t T, int n, int64_t C,
                            cudaStream_t s);
// Per-token part of the post_bda backward: dres (nullable), df (nullable),
// dH_res, dH_post.
cudaError_t launch_post_bwd_tok(const bf16 *dout, const bf16 *res, const bf16 *f,
                                const bf16 *bias, const float *Hres, const float *Hpost,
                                bf16 *dres, bf16 *df, float *dHres, float *dHpost, int64_t T,
                                int n, int64_t C, cudaStream_t s);
// dbias[c] = sum_t sum_i H_post[t][i] dout[t][i][c]; scratch: dbias_ws_bytes.
size_t dbias_ws_bytes(int64_t T, int64_t C);
cudaError_t launch_dbias(const bf16 *dout, const float *Hpost, float *dbias, int64_t T, int n,
                         int64_t C, void *ws, cudaStream_t s);
cudaError_t launch_rms_fwd(const bf16 *x, bf16 *y, float *rstd, int64_t rows, int64_t cols,
                           float eps, cudaStream_t s);
cudaError_t launch_rms_bwd(const bf16 *dy, const bf16 *x, const float *rstd, bf16 *dx,
                           int64_t rows, int64_t cols, float eps, cudaStream_t s);

// k_norm.cu: rmsnorm_residual (h = x + res, y = h rho gamma) and h_aggregate
// fused with that RMSNorm; dgamma through per-block partials (scratch
// norm_ws_bytes(rows, cols)); k_col_sum (grid ceil(cols/32), block 32 x 32)
// adds rows of partials in a fixed order.
__global__ void k_col_sum(const float *__restrict__ part, int64_t nrows, int64_t cols,
                          float *__restrict__ out);
int norm_blocks(int64_t rows);
size_t norm_ws_bytes(int64_t rows, int64_t cols);
cudaError_t launch_rmsr_fwd(const bf16 *x, const bf16 *res, const float *gamma, bf16 *hout,
                            bf16 *y, float *rstd, int64_t rows, int64_t cols, float eps,
                            cudaStream_t s);
cudaError_t launch_rmsr_bwd(const bf16 *dy, const bf16 *dh, const bf16 *x, const bf16 *res,
                            const float *gamma, const float *rstd, bf16 *dx, float *dgamma,
                            int64_t rows, int64_t cols, float eps, void *ws, cudaStream_t s);
cudaError_t launch_aggn_fwd(const bf16 *x, const float *Hpre, const float *gamma, bf16 *y,
                            bf16 *yn, float *rstd, int64_t T, int n, int64_t C, float eps,
                            cudaStream_t s);
cudaError_t launch_aggn_bwd(const bf16 *dyn, const bf16 *dy, const bf16 *x, const float *Hpre,
                            const float *gamma, const float *rstd, bf16 *dx, float *dHpre,
                            float *dgamma, int64_t T, int n, int64_t C, float eps, void *ws,
                            cudaStream_t s);

// k_proj_tc.cu: tensor-core projection partials of the forward
int proj_tc_splits(int64_t T, int n, int64_t K);
void set_batch_invariant(int on);
int batch_invariant();
cudaError_t launch_proj_partials(const bf16 *x, const float *W, int64_t T, int n, int64_t C,
                                 bf16 *Whl, float *upart, float *spart, int *splits_used,
                                 int *fault, cudaStream_t s);

// Width of one partial row of the backward's token sums: dz sums over the
// n*n+2n logits (for db), the three dalpha terms, one pad column.
constexpr int bwd_part_cols(int n) { return n * n + 2 * n + 4; }

// k_bwd_tok.cu: token pass of the layer backward: df and the per-token sums
// dH_res [T][n][n], dH_post [T][n], dH_pre [T][n]
int bwd_tok_blocks(int64_t T);
cudaError_t launch_bwd_tok(const bf16 *dout, const bf16 *x, const bf16 *f, const bf16 *bias,
                           const bf16 *dy, const float *Hpost, int64_t T, int n, int64_t C,
                           bf16 *df, float *dHres, float *dHpost, float *dHpre, cudaStream_t s);

// k_bwd_tc.cu: residual-gradient pass of the backward on the tensor cores
int bwd_tc_du_cols(int n);
int bwd_tc_splits(int64_t T, int n, int64_t C);
// du32 [T][O] fp32 and dub [T] = sum_o |du| serve the exact path of tokens
// whose bf16 product would be too coarse (see k_bwd_tc.cu).
cudaError_t launch_bwd_tc(const bf16 *x, const float *W, const bf16 *du_hl, const float *du32,
                          const float *dub, const float *coef, int64_t T, int n, int64_t C,
                          const bf16 *dout,
                          const bf16 *dy, const float *Hpre, const float *Hres,
                          const float *Hpost, bf16 *dx, float *dWpart, float *dbiaspart,
                          int splits, int *fault, cudaStream_t s);

// k_proj.cu
size_t proj_fwd_ws_bytes(int64_t T, int n, int64_t C);
// Rows of W_hl: W as three bf16 terms (hi, lo, lo2: 3O rows), padded with
// zero rows to the MMA's N granularity of 16 (80 at n = 4, 240 at n = 8).
__host__ __device__ constexpr int w_split_rows(int n) { return (3 * (n * n + 2 * n) + 15) / 16 * 16; }
// W [K][O] fp32 -> W_hl [w_split_rows(n)][K] bf16: rows o = bf16(W[:,o]),
// rows O+o = bf16 of the remainder, rows 2O+o = bf16 of what is left, then
// zero rows
cudaError_t launch_w_split(const float *W, bf16 *Whl, int n, int64_t K, cudaStream_t s);
// compute_h forward from S split partials upart [S][T][O], spart [S][T]
cudaError_t launch_compute_h_parts(const float *upart, const float *spart, int S,
                                   const float *alpha, const float *b, int64_t T, int n,
                                   int64_t C, int iters, float eps_sk, float eps_rms, float *Hpre,
                                   float *Hpost, float *Hres, float *u_save, float *r_save,
                                   cudaStream_t s);
// selftest.cu: a bounded wait that runs out after `limit` cycles
cudaError_t launch_selftest_wait(long long limit, int *fault, cudaStream_t s);
// k_post_proj.cu: the post-mix of a layer fused with the next layer's
// proj_rms_compute_h forward on its output (workspace post_proj_ws_bytes).
size_t post_proj_ws_bytes(int64_t T, int n, int64_t C);
cudaError_t launch_post_proj_fwd(const bf16 *res, const bf16 *f, const bf16 *bias,
                                 const float *Hres, const float *Hpost, const float *Wn,
                                 const float *alphan, const float *bn, int64_t T, int n,
                                 int64_t C, int iters, float eps_sk, float eps_rms, bf16 *out,
                                 float *Hpre_n, float *Hpost_n, float *Hres_n, float *u_save_n,
                                 float *r_save_n, void *ws, int *fault, cudaStream_t s);
cudaError_t launch_proj_fwd(const bf16 *x, const float *W, const float *alpha, const float *b,
                            int64_t T, int n, int64_t C, int iters, float eps_sk, float eps_rms,
                            float *Hpre, float *Hpost, float *Hres, float *u_save, float *r_save,
                            void *ws, int *fault, cudaStream_t s);
// Backward of proj_rms_compute_h (standalone op); workspace proj_bwd_ws_bytes.
size_t proj_bwd_ws_bytes(int64_t T, int n, int64_t C);
cudaError_t launch_proj_bwd(const float *dHpre, const float *dHpost, const float *dHres,
                            const bf16 *x, const float *W, const float *alpha, const float *b,
                            const float *u_save, const float *r_save, int64_t T, int n,
                            int64_t C, int iters, float eps_sk, float eps_rms, bf16 *dx,
                            float *dW, float *dalpha, float *db, void *ws, int *fault,
                            cudaStream_t s);
// Layer backward (two passes over HBM): the token pass (post_bda and
// aggregate reductions, df), the compute_h backward, then the
// residual-gradient pass dx = H_res dout + H_pre dy + du W^T + coef x with
// dW and dbias.  Workspace proj_bwd_ws_bytes.
// Channel-sharded proj_rms_compute_h: a shard's partial sums u [T][O], s [T]
// (scratch proj_fwd_ws_bytes(T, n, Cs)); compute_h from the totals; the
// per-token backward coefficients du, coef with dalpha, db (scratch
// compute_h_bwd_ws_bytes); a shard's dx and dW (scratch proj_bwd_ws_bytes(T, n, Cs)).
cudaError_t launch_proj_partial_sums(const bf16 *x, const float *W, int64_t T, int n, int64_t Cs,
                                     float *u, float *s_out, void *ws, int *fault, cudaStream_t s);
cudaError_t launch_compute_h_fwd(const float *u, const float *s_tot, int64_t K,
                                 const float *alpha, const float *b, int64_t T, int n, int iters,
                                 float eps_sk, float eps_rms, float *Hpre, float *Hpost,
                                 float *Hres, float *r_save, cudaStream_t s);
size_t compute_h_bwd_ws_bytes(int64_t T, int n);
cudaError_t launch_compute_h_bwd(const float *dHpre, const float *dHpost, const float *dHres,
                                 const float *u, const float *s_tot, int64_t K,
                                 const float *alpha, const float *b, int64_t T, int n, int iters,
                                 float eps_sk, float eps_rms, float *du, float *coef,
                                 float *dalpha, float *db, void *ws, cudaStream_t s);
cudaError_t launch_proj_partial_bwd(const bf16 *x, const float *W, const float *du,
                                    const float *coef, int64_t T, int n, int64_t Cs, bf16 *dx,
                                    float *dW, void *ws, int *fault, cudaStream_t s);
cudaError_t launch_layer_bwd(const bf16 *dout, const bf16 *dy, const bf16 *x, const float *W,
                             const float *alpha, const float *b, const bf16 *f,
                             const bf16 *bias, const float *Hpre, const float *Hpost,
                             const float *Hres, const float *u_save, const float *r_save,
                             int64_t T, int n, int64_t C, int iters, float eps_sk,
                             float eps_rms, bf16 *dx, bf16 *df, float *dW, float *dalpha,
                             float *db, float *dbias, void *ws, int *fault, cudaStream_t s);

// k_pinned.cu: the bit-reproducible mode (pinned reduction trees, n = 4)
void set_pinned(int on);
int pinned();
size_t pin_bwd_ws_bytes(int64_t T);
cudaError_t launch_pin_sinkhorn_fwd(const float *lg, float *P, int64_t M, int iters, float eps,
                                    cudaStream_t s);
cudaError_t launch_pin_sinkhorn_bwd(const float *dP, const float *lg, float *dl, int64_t M,
                                    int iters, float eps, cudaStream_t s);
cudaError_t launch_pin_proj_fwd(const bf16 *x, const float *W, const float *alpha, const float *b,
                                int64_t T, int64_t C, int iters, float eps_sk, float eps_rms,
                                float *Hpre, float *Hpost, float *Hres, float *u_save,
                                float *r_save, cudaStream_t s);
cudaError_t launch_pin_proj_bwd(const float *dHpre, const float *dHpost, const float *dHres,
                                const bf16 *x, const float *W, const float *alpha, const float *b,
                                int64_t T, int64_t C, int iters, float eps_sk, float eps_rms,
                                bf16 *dx, float *dW, float *dalpha, float *db, void *ws,
                                cudaStream_t s);
cudaError_t launch_pin_agg_fwd(const bf16 *x, const float *Hpre, bf16 *y, int64_t T, int64_t C,
                               cudaStream_t s);
cudaError_t launch_pin_agg_bwd(const bf16 *dy, const bf16 *x, const float *Hpre, bf16 *dx,
                               float *dHpre, int64_t T, int64_t C, cudaStream_t s);
cudaError_t launch_pin_post_fwd(const bf16 *res, const bf16 *f, const bf16 *bias,
                                const float *Hres, const float *Hpost, bf16 *out, int64_t T,
                                int64_t C, cudaStream_t s);
cudaError_t launch_pin_post_bwd(const bf16 *dout, const bf16 *res, const bf16 *f,
                                const bf16 *bias, const float *Hres, const float *Hpost,
                                bf16 *dres, bf16 *df, float *dbias, float *dHres, float *dHpost,
                                int64_t T, int64_t C, cudaStream_t s);
cudaError_t launch_pin_layer_fwd(const bf16 *x, const float *W, const float *alpha,
                                 const float *b, const bf16 *f, const bf16 *bias, int64_t T,
                                 int64_t C, int iters, float eps_sk, float eps_rms, float *Hpre,
                                 float *Hpost, float *Hres, float *u_save, float *r_save, bf16 *y,
                                 bf16 *out, cudaStream_t s);
cudaError_t launch_pin_layer_bwd(const bf16 *dout, const bf16 *dy, const bf16 *x, const float *W,
                                 const float *alpha, const float *b, const bf16 *f,
                                 const bf16 *bias, const float *Hpre, const float *Hpost,
                                 const float *Hres, int64_t T, int64_t C, int iters, float eps_sk,
                                 float eps_rms, bf16 *dx, bf16 *df, float *dW, float *dalpha,
                                 float *db, float *dbias, void *ws, cudaStream_t s);

}  // namespace mhc
