// Sinkhorn-Knopp on n x n matrices held by groups of n lanes.
//
// Definition (rwkv-ops mhu_ffi.cu SinkhornFwdHost/SinkhornBwdHost; Megatron-Core
// fused_mhc_kernels fused_sinkhorn): A = exp(z); then `iters` times divide
// every row by (row sum + eps), then every column by (column sum + eps).  The
// backward is the exact gradient of that unrolled map.
//
// Layout in registers: a group of N consecutive lanes (N in {4, 8}, aligned
// to N) holds one matrix; lane i of the group holds row i as N floats.  Row
// sums are local; column sums are a butterfly over the group's lanes.  A
// division by a denominator is a multiplication by the hardware's
// approximate reciprocal (rcp.approx, within an ulp of 1/d; one per row
// step, one per column), as in the one-thread-per-matrix form below.  All 32
// lanes of the warp must call these functions together (the shuffles use
// the full mask); a group without work runs on dummy data.
#pragma once

#include "common.cuh"

namespace mhc {

template <int N>
__device__ __forceinline__ void sk_colsum(const float (&v)[N], float (&cs)[N])
{
#pragma unroll
    for (int j = 0; j < N; ++j) cs[j] = v[j];
#pragma unroll
    for (int m = 1; m < N; m <<= 1)
#pragma unroll
        for (int j = 0; j < N; ++j) cs[j] += __shfl_xor_sync(kFull, cs[j], m);
}

// Forward.  a: in exp(z) row, out the row of P.  If `store` is not null the
// denominators of every step are kept for the backward: store[(2k)*stride]
// is (this lane's row sum + eps) at the row step of iteration k, and
// store[(2k+1)*stride] is (column (lane % N)'s sum + eps) at its column step.
template <int N>
__device__ __forceinline__ void sk_forward(float (&a)[N], int iters, float eps, float *store,
                                           int stride)
{
    const int i = threadIdx.x & (N - 1);
    for (int k = 0; k < iters; ++k) {
        float rs = 0.f;
#pragma unroll
        for (int j = 0; j < N; ++j) rs += a[j];
        const float rd = rs + eps;
        const float rinv = rcp_approx(rd);
#pragma unroll
        for (int j = 0; j < N; ++j) a[j] *= rinv;
        float cs[N];
        sk_colsum<N>(a, cs);
        float cd_mine = 0.f;
#pragma unroll
        for (int j = 0; j < N; ++j) {
            const float cd = cs[j] + eps;
            a[j] *= rcp_approx(cd);
            if (j == i) cd_mine = cd;
        }
        if (store) {
            store[(2 * k) * stride] = rd;
            store[(2 * k + 1) * stride] = cd_mine;
        }
    }
}

// Backward.  On entry g holds this lane's row of dL/dP, a the row of P (the
// forward output) and e the row of exp(z); `store` the denominators written
// by sk_forward.  On exit g holds the row of dL/dz.  a is consumed: walking
// the steps in reverse, each intermediate matrix is rebuilt by multiplying
// back the stored denominator.
//   column step Y = X / cd_j:  dX[i][j] = (dY[i][j] - sum_i' dY[i'][j] Y[i'][j]) / cd_j
//   row step    Y = X / rd_i:  dX[i][j] = (dY[i][j] - sum_j' dY[i][j'] Y[i][j']) / rd_i
template <int N>
__device__ __forceinline__ void sk_backward(float (&g)[N], float (&a)[N], const float (&e)[N],
                                            int iters, const float *store, int stride)
{
    const int lane = threadIdx.x & (kWarp - 1);
    const int base = lane & ~(N - 1);
    for (int k = iters - 1; k >= 0; --k) {
        const float rd = store[(2 * k) * stride];
        const float cd_mine = store[(2 * k + 1) * stride];
        float ga[N], dot[N], cd[N];
#pragma unroll
        for (int j = 0; j < N; ++j) ga[j] = g[j] * a[j];
        sk_colsum<N>(ga, dot);
#pragma unroll
        for (int j = 0; j < N; ++j) cd[j] = __shfl_sync(kFull, cd_mine, base + j);
#pragma unroll
        for (int j = 0; j < N; ++j) {
            g[j] = (g[j] - dot[j]) * rcp_approx(cd[j]);
            a[j] = a[j] * cd[j];
        }
        float rdot = 0.f;
#pragma unroll
        for (int j = 0; j < N; ++j) rdot += g[j] * a[j];
        const float rinv = rcp_approx(rd);
#pragma unroll
        for (int j = 0; j < N; ++j) {
            g[j] = (g[j] - rdot) * rinv;
            a[j] = a[j] * rd;
        }
    }
#pragma unroll
    for (int j = 0; j < N; ++j) g[j] = g[j] * e[j];
}

// ---------------------------------------------------------------------------
// ---------------------------------------------------------------------------
// n = 4 with one thread per matrix, the 16 entries in registers.  Row and
// column sums are local (four independent chains per half-step instead of a
// shuffle butterfly): row sums ((a0 + a1) + a2) + a3, column sums
// (a0 + a1) + (a2 + a3), every product and sum explicitly rounded.  A
// division by a denominator is a multiplication by the hardware's
// approximate reciprocal (rcp.approx, within an ulp): with one thread per
// matrix or token there are few warps per SM, so these kernels are bound by
// their instruction count, of which the correctly rounded reciprocal took
// half.  The backward reads the 8 denominators of every iteration that the
// forward stored at store[(8k + d) * stride].
// ---------------------------------------------------------------------------
// store: denominators of iteration k at store[(8k + d) * stride], d < 4 the
// row steps', d >= 4 the column steps' (or null)
__device__ __forceinline__ void sk4_forward(float (&a)[4][4], int iters, float eps, float *store,
                                            int stride)
{
    for (int k = 0; k < iters; ++k) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float rd =
                __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(a[i][0], a[i][1]), a[i][2]), a[i][3]), eps);
            const float rinv = rcp_approx(rd);
#pragma unroll
            for (int j = 0; j < 4; ++j) a[i][j] = __fmul_rn(a[i][j], rinv);
            if (store) store[(8 * k + i) * stride] = rd;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float cd = __fadd_rn(
                __fadd_rn(__fadd_rn(a[0][j], a[1][j]), __fadd_rn(a[2][j], a[3][j])), eps);
            const float cinv = rcp_approx(cd);
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i][j] = __fmul_rn(a[i][j], cinv);
            if (store) store[(8 * k + 4 + j) * stride] = cd;
        }
    }
}

// Backward, walking the steps in reverse (the gradient sk_backward forms):
//   column step Y = X / cd_j:  dX[i][j] = (dY[i][j] - sum_i' dY[i'][j] Y[i'][j]) / cd_j
//   row step    Y = X / rd_i:  dX[i][j] = (dY[i][j] - sum_j' dY[i][j'] Y[i][j']) / rd_i
// On entry g = dL/dP, a = P, e = exp(z); on exit g = dL/dz (a consumed).
__device__ __forceinline__ void sk4_backward(float (&g)[4][4], float (&a)[4][4],
                                             const float (&e)[4][4], int iters, const float *store,
                                             int stride)
{
    for (int k = iters - 1; k >= 0; --k) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float cd = store[(8 * k + 4 + j) * stride];
            float ga[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) ga[i] = __fmul_rn(g[i][j], a[i][j]);
            const float dot = __fadd_rn(__fadd_rn(ga[0], ga[1]), __fadd_rn(ga[2], ga[3]));
            const float cinv = rcp_approx(cd);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                g[i][j] = __fmul_rn(__fsub_rn(g[i][j], dot), cinv);
                a[i][j] = __fmul_rn(a[i][j], cd);
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float rd = store[(8 * k + i) * stride];
            float rdot = __fmul_rn(g[i][0], a[i][0]);
#pragma unroll
            for (int j = 1; j < 4; ++j) rdot = fmaf(g[i][j], a[i][j], rdot);
            const float rinv = rcp_approx(rd);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                g[i][j] = __fmul_rn(__fsub_rn(g[i][j], rdot), rinv);
                a[i][j] = __fmul_rn(a[i][j], rd);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) g[i][j] = __fmul_rn(g[i][j], e[i][j]);
}

}  // namespace mhc
