// RMSNorm with a residual fork and a learnable weight (rmsnorm_residual), and
// h_aggregate fused with that RMSNorm.
//
// Definitions (RL-Kernel PR #383, PR body tasks P1-5 "RMSNorm + residual
// fork" and P1-8 "cross-rank dgamma"; the follow-up commit on exposing the
// pre-normalization intermediate):
//   rmsnorm_residual:  h = x + res (res optional), rho = 1/sqrt(sum_c h^2/C + eps),
//                      y = h rho gamma (gamma optional);  h is returned as well.
//     backward:        g = dy gamma;  dx = dres = dh + rho g - rho^3 h (sum_c g h)/C,
//                      dgamma[c] = sum_t dy h rho.
//   aggregate + norm:  y = sum_i H_pre[i] x_i (Megatron-Core fused_h_aggregate),
//                      yn = y rho gamma;  backward: dy_total = dy + the RMSNorm
//                      backward of dyn, then dx_i = H_pre[i] dy_total and
//                      dH_pre[i] = sum_c dy_total x_i.
//
// Layout of the work: one block per row at a time (rows strided over a fixed
// grid); thread tid owns the 8-channel chunks j = tid + NT q (q < CPT) of
// every row, so the row reductions are block sums in a fixed order and the
// dgamma partial of a block stays in its threads' registers.  The grid is a
// fixed function of the shape, so the per-block dgamma partials and their
// final sum (k_col_sum, ascending block order) are deterministic.
#include "launch.h"

namespace mhc {

// Sums of NV values over the block; every thread receives the totals
// (warp butterflies, then the warps' partials in ascending warp order).
template <int NV>
__device__ __forceinline__ void rb_sum(float (&v)[NV], float *red /* [NV * 32] */)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int k = 0; k < NV; ++k) v[k] = warp_sum(v[k]);
    if (lane == 0)
#pragma unroll
        for (int k = 0; k < NV; ++k) red[k * 32 + w] = v[k];
    __syncthreads();
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        float s = 0.f;
        for (int i = 0; i < nw; ++i) s += red[k * 32 + i];
        v[k] = s;
    }
    __syncthreads();
}

__device__ __forceinline__ void load_gamma8(const float *gamma, int64_t j, float (&g)[8])
{
    if (gamma) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(gamma + j * 8));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(gamma + j * 8 + 4));
        g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
        g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) g[e] = 1.f;
    }
}

__device__ __forceinline__ void store_part8(float *p, const float (&v)[8])
{
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

// ---------------------------------------------------------------------------
// rmsnorm_residual forward
// ---------------------------------------------------------------------------
template <int CPT>
__global__ void __launch_bounds__(512)
    k_rmsr_fwd(const bf16 *__restrict__ x, const bf16 *__restrict__ res,
               const float *__restrict__ gamma, bf16 *__restrict__ hout, bf16 *__restrict__ y,
               float *__restrict__ rstd, int64_t rows, int64_t C8, float inv_cols, float eps)
{
    pdl_wait();
    __shared__ float red[32];
    const int tid = threadIdx.x, NT = blockDim.x;
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        float h[CPT][8];
        float ss[1] = {0.f};
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const int64_t j = tid + int64_t(NT) * q;
#pragma unroll
            for (int e = 0; e < 8; ++e) h[q][e] = 0.f;
            if (j < C8) {
                unpack8(ld_stream(x + (r * C8 + j) * 8), h[q]);
                if (res) {
                    float v[8];
                    unpack8(ld_stream(res + (r * C8 + j) * 8), v);
#pragma unroll
                    for (int e = 0; e < 8; ++e) h[q][e] += v[e];
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) ss[0] = fmaf(h[q][e], h[q][e], ss[0]);
            }
        }
        rb_sum<1>(ss, red);
        const float rho = rsqrtf(ss[0] * inv_cols + eps);
        if (rstd && tid == 0) rstd[r] = rho;
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const int64_t j = tid + int64_t(NT) * q;
            if (j < C8) {
                if (hout) st_stream(hout + (r * C8 + j) * 8, pack8(h[q]));
                float g[8], o[8];
                load_gamma8(gamma, j, g);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = h[q][e] * rho * g[e];
                st_stream(y + (r * C8 + j) * 8, pack8(o));
            }
        }
    }
}

// ---------------------------------------------------------------------------
// rmsnorm_residual backward (dx, and per-block dgamma partials)
// ---------------------------------------------------------------------------
template <int CPT>
__global__ void __launch_bounds__(512)
    k_rmsr_bwd(const bf16 *__restrict__ dy, const bf16 *__restrict__ dh,
               const bf16 *__restrict__ x, const bf16 *__restrict__ res,
               const float *__restrict__ gamma, const float *__restrict__ rstd,
               bf16 *__restrict__ dx, float *__restrict__ dgpart, int64_t rows, int64_t C8,
               float inv_cols, float eps)
{
    pdl_wait();
    __shared__ float red[64];
    const int tid = threadIdx.x, NT = blockDim.x;
    float acc[CPT][8];
#pragma unroll
    for (int q = 0; q < CPT; ++q)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[q][e] = 0.f;
    // the row's inputs stay packed (bf16) across the block sum; h = x + res
    // is re-formed from them in fp32 where it is used
    auto fork = [&](const uint4 xv, const uint4 rv, float (&h)[8]) {
        unpack8(xv, h);
        if (res) {
            float v[8];
            unpack8(rv, v);
#pragma unroll
            for (int e = 0; e < 8; ++e) h[e] += v[e];
        }
    };
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        uint4 xv[CPT], rv[CPT], dv[CPT];
        float sums[2] = {0.f, 0.f};  // sum g h, sum h^2
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const int64_t j = tid + int64_t(NT) * q;
            xv[q] = rv[q] = dv[q] = make_uint4(0, 0, 0, 0);
            if (j < C8) {
                xv[q] = ld_stream(x + (r * C8 + j) * 8);
                if (res) rv[q] = ld_stream(res + (r * C8 + j) * 8);
                dv[q] = ld_stream(dy + (r * C8 + j) * 8);
            }
        }
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const int64_t j = tid + int64_t(NT) * q;
            if (j < C8) {
                float h[8], d[8], g[8];
                fork(xv[q], rv[q], h);
                unpack8(dv[q], d);
                load_gamma8(gamma, j, g);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    sums[0] = fmaf(d[e] * g[e], h[e], sums[0]);
                    sums[1] = fmaf(h[e], h[e], sums[1]);
                }
            }
        }
        rb_sum<2>(sums, red);
        const float rho = rstd ? __ldg(rstd + r) : rsqrtf(sums[1] * inv_cols + eps);
        const float k3 = rho * rho * rho * sums[0] * inv_cols;
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const int64_t j = tid + int64_t(NT) * q;
            if (j < C8) {
                float h[8], d[8], g[8], o[8];
                fork(xv[q], rv[q], h);
                unpack8(dv[q], d);
                load_gamma8(gamma, j, g);
                if (dh)
                    unpack8(ld_stream(dh + (r * C8 + j) * 8), o);
                else
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    o[e] += rho * (d[e] * g[e]) - k3 * h[e];
                    acc[q][e] = fmaf(d[e] * h[e], rho, acc[q][e]);
                }
                st_stream(dx + (r * C8 + j) * 8, pack8(o));
            }
        }
    }
    if (dgpart)
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const int64_t j = tid + int64_t(NT) * q;
            if (j < C8) store_part8(dgpart + (int64_t(blockIdx.x) * C8 + j) * 8, acc[q]);
        }
}

// ---------------------------------------------------------------------------
// h_aggregate + weighted RMSNorm, forward: y = sum_i H_pre[i] x_i (bf16 out,
// optional), yn = y rho gamma from the fp32 y
// ---------------------------------------------------------------------------
template <int N, int CPT>
__global__ void __launch_bounds__(512)
    k_aggn_fwd(const bf16 *__restrict__ x, const float *__restrict__ Hpre,
               const float *__restrict__ gamma, bf16 *__restrict__ y, bf16 *__restrict__ yn,
               float *__restrict__ rstd, int64_t T, int64_t C8, float inv_cols, float eps)
{
    pdl_wait();
    __shared__ float red[32];
    const int tid = threadIdx.x, NT = blockDim.x;
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        float hp[N];
#pragma unroll
        for (int i = 0; i < N; ++i) hp[i] = __ldg(Hpre + t * N + i);
        float yv[CPT][8];
        float ss[1] = {0.f};
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const int64_t j = tid + int64_t(NT) * q;
#pragma unroll
            for (int e = 0; e < 8; ++e) yv[q][e] = 0.f;
            if (j < C8) {
#pragma unroll
                for (int i = 0; i < N; ++i) {
                    float v[8];
                    unpack8(ld_stream(x + ((t * N + i) * C8 + j) * 8), v);
#pragma unroll
                    for (int e = 0; e < 8; ++e) yv[q][e] = fmaf(hp[i], v[e], yv[q][e]);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) ss[0] = fmaf(yv[q][e], yv[q][e], ss[0]);
            }
        }
        rb_sum<1>(ss, red);
        const float rho = rsqrtf(ss[0] * inv_cols + eps);
        if (rstd && tid == 0) rstd[t] = rho;
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const int64_t j = tid + int64_t(NT) * q;
            if (j < C8) {
                if (y) st_stream(y + (t * C8 + j) * 8, pack8(yv[q]));
                float g[8], o[8];
                load_gamma8(gamma, j, g);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = yv[q][e] * rho * g[e];
                st_stream(yn + (t * C8 + j) * 8, pack8(o));
            }
        }
    }
}

// ---------------------------------------------------------------------------
// h_aggregate + weighted RMSNorm, backward: dx, dH_pre per token, per-block
// dgamma partials.  x is read once per token and kept in registers.
// ---------------------------------------------------------------------------
template <int N, int CPT>
__global__ void __launch_bounds__(512)
    k_aggn_bwd(const bf16 *__restrict__ dyn, const bf16 *__restrict__ dy,
               const bf16 *__restrict__ x, const float *__restrict__ Hpre,
               const float *__restrict__ gamma, const float *__restrict__ rstd,
               bf16 *__restrict__ dx, float *__restrict__ dHpre, float *__restrict__ dgpart,
               int64_t T, int64_t C8, float inv_cols, float eps)
{
    pdl_wait();
    // x stays in registers between the two phases when it is small enough,
    // else the second phase reads it again (an L2 hit); y is re-formed from
    // x in the second phase
    constexpr bool KEEP = N * CPT <= 8;
    __shared__ float red[N * 32];
    const int tid = threadIdx.x, NT = blockDim.x;
    float acc[CPT][8];
#pragma unroll
    for (int q = 0; q < CPT; ++q)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[q][e] = 0.f;
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        float hp[N];
#pragma unroll
        for (int i = 0; i < N; ++i) hp[i] = __ldg(Hpre + t * N + i);
        uint4 xr[KEEP ? CPT : 1][N], gv[CPT];
        float sums[2] = {0.f, 0.f};  // sum g y, sum y^2
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const int64_t j = tid + int64_t(NT) * q;
            gv[q] = make_uint4(0, 0, 0, 0);
            if (j < C8) {
                float yv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < N; ++i) {
                    const uint4 xv = ld_stream(x + ((t * N + i) * C8 + j) * 8);
                    if (KEEP) xr[KEEP ? q : 0][i] = xv;
                    float v[8];
                    unpack8(xv, v);
#pragma unroll
                    for (int e = 0; e < 8; ++e) yv[e] = fmaf(hp[i], v[e], yv[e]);
                }
                gv[q] = ld_stream(dyn + (t * C8 + j) * 8);
                float gd[8], g[8];
                unpack8(gv[q], gd);
                load_gamma8(gamma, j, g);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    sums[0] = fmaf(gd[e] * g[e], yv[e], sums[0]);
                    sums[1] = fmaf(yv[e], yv[e], sums[1]);
                }
            }
        }
        rb_sum<2>(sums, red);
        const float rho = rstd ? __ldg(rstd + t) : rsqrtf(sums[1] * inv_cols + eps);
        const float k3 = rho * rho * rho * sums[0] * inv_cols;
        float pd[N];
#pragma unroll
        for (int i = 0; i < N; ++i) pd[i] = 0.f;
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const int64_t j = tid + int64_t(NT) * q;
            if (j < C8) {
                uint4 xq[N];
                float yv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < N; ++i) {
                    xq[i] = KEEP ? xr[KEEP ? q : 0][i] : ld_stream(x + ((t * N + i) * C8 + j) * 8);
                    float v[8];
                    unpack8(xq[i], v);
#pragma unroll
                    for (int e = 0; e < 8; ++e) yv[e] = fmaf(hp[i], v[e], yv[e]);
                }
                float g[8], gd[8], dt[8];
                load_gamma8(gamma, j, g);
                unpack8(gv[q], gd);
                if (dy)
                    unpack8(ld_stream(dy + (t * C8 + j) * 8), dt);
                else
#pragma unroll
                    for (int e = 0; e < 8; ++e) dt[e] = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    dt[e] += rho * (gd[e] * g[e]) - k3 * yv[e];
                    acc[q][e] = fmaf(gd[e] * yv[e], rho, acc[q][e]);
                }
#pragma unroll
                for (int i = 0; i < N; ++i) {
                    float v[8], o[8];
                    unpack8(xq[i], v);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        pd[i] = fmaf(dt[e], v[e], pd[i]);
                        o[e] = hp[i] * dt[e];
                    }
                    st_stream(dx + ((t * N + i) * C8 + j) * 8, pack8(o));
                }
            }
        }
        rb_sum<N>(pd, red);
        if (tid == 0)
#pragma unroll
            for (int i = 0; i < N; ++i) dHpre[t * N + i] = pd[i];
    }
    if (dgpart)
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
            const int64_t j = tid + int64_t(NT) * q;
            if (j < C8) store_part8(dgpart + (int64_t(blockIdx.x) * C8 + j) * 8, acc[q]);
        }
}

// out[c] = sum_b part[b][c] in a fixed order: a 32 x 32 block covers 32
// columns; thread (x, y) adds rows b = y, y + 32, ... in ascending order,
// then the 32 row-group sums of a column are added in ascending y.
// Launch: grid ceil(cols / 32), block (32, 32).
__global__ void __launch_bounds__(1024)
    k_col_sum(const float *__restrict__ part, int64_t nrows, int64_t cols,
              float *__restrict__ out)
{
    pdl_wait();
    __shared__ float red[32][33];
    const int64_t c = int64_t(blockIdx.x) * 32 + threadIdx.x;
    float s = 0.f;
    if (c < cols)
        for (int64_t b = threadIdx.y; b < nrows; b += 32) s += part[b * cols + c];
    red[threadIdx.y][threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.y == 0 && c < cols) {
        float t = 0.f;
        for (int g = 0; g < 32; ++g) t += red[g][threadIdx.x];
        out[c] = t;
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// Chunks per thread and threads per block for rows of C8 chunks (C8 <= 4096):
// four chunks per thread where the row has more than 256 chunks, so that a
// 7B-scale row (512 chunks) is a 128-thread block and four rows are in
// flight per SM.
static void norm_shape(int64_t C8, int *cpt, int *nt)
{
    int c = C8 > 256 ? 4 : (C8 > 128 ? 2 : 1);
    if ((C8 + c - 1) / c > 512) c = 8;
    int64_t t = (C8 + c - 1) / c;
    t = (t + 31) / 32 * 32;
    *cpt = c;
    *nt = int(t);
}

int norm_blocks(int64_t rows)
{
    const int64_t cap = int64_t(kSplitSms) * 8;
    return int(rows < cap ? (rows > 0 ? rows : 1) : cap);
}

size_t norm_ws_bytes(int64_t rows, int64_t cols)
{
    return ws_align(size_t(norm_blocks(rows)) * size_t(cols) * 4);
}

#define MHC_NORM_CPT_SWITCH(CPT_VAR, ...)                                                         \
    switch (CPT_VAR) {                                                                           \
    case 1: { constexpr int CPT = 1; __VA_ARGS__; } break;                                       \
    case 2: { constexpr int CPT = 2; __VA_ARGS__; } break;                                       \
    case 4: { constexpr int CPT = 4; __VA_ARGS__; } break;                                       \
    default: { constexpr int CPT = 8; __VA_ARGS__; } break;                                      \
    }

cudaError_t launch_rmsr_fwd(const bf16 *x, const bf16 *res, const float *gamma, bf16 *hout,
                            bf16 *y, float *rstd, int64_t rows, int64_t cols, float eps,
                            cudaStream_t s)
{
    const int64_t C8 = cols / 8;
    int cpt, nt;
    norm_shape(C8, &cpt, &nt);
    const unsigned g = unsigned(norm_blocks(rows));
    const float ic = 1.0f / float(cols);
    MHC_PROF("k_rmsr_fwd", s);
    MHC_NORM_CPT_SWITCH(cpt, launch_k(k_rmsr_fwd<CPT>, dim3(g), dim3(nt), 0, s, x, res, gamma, hout, y, rstd, rows,
                                                               C8, ic, eps));
    return cudaGetLastError();
}

cudaError_t launch_rmsr_bwd(const bf16 *dy, const bf16 *dh, const bf16 *x, const bf16 *res,
                            const float *gamma, const float *rstd, bf16 *dx, float *dgamma,
                            int64_t rows, int64_t cols, float eps, void *ws, cudaStream_t s)
{
    const int64_t C8 = cols / 8;
    int cpt, nt;
    norm_shape(C8, &cpt, &nt);
    const int nb = norm_blocks(rows);
    const float ic = 1.0f / float(cols);
    float *part = dgamma ? static_cast<float *>(ws) : nullptr;
    {
        MHC_PROF("k_rmsr_bwd", s);
        MHC_NORM_CPT_SWITCH(cpt, launch_k(k_rmsr_bwd<CPT>, dim3(unsigned(nb)), dim3(nt), 0, s, 
                                     dy, dh, x, res, gamma, rstd, dx, part, rows, C8, ic, eps));
    }
    if (dgamma) {
        MHC_PROF("k_col_sum", s);
        launch_k(k_col_sum, dim3(unsigned((cols + 31) / 32)), dim3(dim3(32, 32)), 0, s, part, nb, cols, dgamma);
    }
    return cudaGetLastError();
}

cudaError_t launch_aggn_fwd(const bf16 *x, const float *Hpre, const float *gamma, bf16 *y,
                            bf16 *yn, float *rstd, int64_t T, int n, int64_t C, float eps,
                            cudaStream_t s)
{
    const int64_t C8 = C / 8;
    int cpt, nt;
    norm_shape(C8, &cpt, &nt);
    const unsigned g = unsigned(norm_blocks(T));
    const float ic = 1.0f / float(C);
    MHC_PROF("k_aggn_fwd", s);
    if (n == 4) {
        MHC_NORM_CPT_SWITCH(cpt, launch_k(k_aggn_fwd<4, CPT>, dim3(g), dim3(nt), 0, s, x, Hpre, gamma, y, yn, rstd,
                                                                      T, C8, ic, eps));
    } else {
        MHC_NORM_CPT_SWITCH(cpt, launch_k(k_aggn_fwd<8, CPT>, dim3(g), dim3(nt), 0, s, x, Hpre, gamma, y, yn, rstd,
                                                                      T, C8, ic, eps));
    }
    return cudaGetLastError();
}

cudaError_t launch_aggn_bwd(const bf16 *dyn, const bf16 *dy, const bf16 *x, const float *Hpre,
                            const float *gamma, const float *rstd, bf16 *dx, float *dHpre,
                            float *dgamma, int64_t T, int n, int64_t C, float eps, void *ws,
                            cudaStream_t s)
{
    const int64_t C8 = C / 8;
    int cpt, nt;
    norm_shape(C8, &cpt, &nt);
    const int nb = norm_blocks(T);
    const float ic = 1.0f / float(C);
    float *part = dgamma ? static_cast<float *>(ws) : nullptr;
    {
        MHC_PROF("k_aggn_bwd", s);
        if (n == 4) {
            MHC_NORM_CPT_SWITCH(cpt, launch_k(k_aggn_bwd<4, CPT>, dim3(unsigned(nb)), dim3(nt), 0, s, 
                                         dyn, dy, x, Hpre, gamma, rstd, dx, dHpre, part, T, C8,
                                         ic, eps));
        } else {
            MHC_NORM_CPT_SWITCH(cpt, launch_k(k_aggn_bwd<8, CPT>, dim3(unsigned(nb)), dim3(nt), 0, s, 
                                         dyn, dy, x, Hpre, gamma, rstd, dx, dHpre, part, T, C8,
                                         ic, eps));
        }
    }
    if (dgamma) {
        MHC_PROF("k_col_sum", s);
        launch_k(k_col_sum, dim3(unsigned((C + 31) / 32)), dim3(dim3(32, 32)), 0, s, part, nb, C, dgamma);
    }
    return cudaGetLastError();
}

}  // namespace mhc
