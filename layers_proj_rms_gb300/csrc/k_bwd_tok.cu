// Token pass of the mHC layer backward: one read of dout, x, f and dy.
//
// One warp per token streams the token's rows once and forms
//   dH_res[j][i] = sum_c x[j][c] dout[i][c]      dH_post[i] = sum_c dout[i][c] (f[c] + bias[c])
//   dH_pre[i]    = sum_c dy[c] x[i][c]           df[c]      = sum_i H_post[i] dout[i][c]
// (Megatron-Core fused_mhc_kernels _torch_h_post_bda_bwd and
// _torch_h_aggregate_bwd: the post_bda and aggregate reductions of one token
// share its read of x).  The per-token sums go to k_compute_h_bwd, which runs
// the Sinkhorn backward for a group of tokens per warp.
#include "launch.h"

namespace mhc {

constexpr int kTokWarps = 8;
#ifndef MHC_TOK_U
#define MHC_TOK_U 2
#endif
#ifndef MHC_TOK_MINB
#define MHC_TOK_MINB 1
#endif

// U: 8-channel chunks per lane in flight per step
template <int N, int U>
__global__ void __launch_bounds__(32 * kTokWarps, N == 4 ? MHC_TOK_MINB : 1)
    k_bwd_tok(const bf16 *__restrict__ dout, const bf16 *__restrict__ x,
              const bf16 *__restrict__ f, const bf16 *__restrict__ bias,
              const bf16 *__restrict__ dy, const float *__restrict__ Hpost, int64_t T,
              int64_t C8, bf16 *__restrict__ df, float *__restrict__ dHres,
              float *__restrict__ dHpost, float *__restrict__ dHpre)
{
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t warps = int64_t(gridDim.x) * kTokWarps;
    for (int64_t t = int64_t(blockIdx.x) * kTokWarps + warp; t < T; t += warps) {
        // element pairs in f32x2 arithmetic: the running sums are pairs (even
        // and odd channels of a chunk), added together once per token
        f32x2 hp2[N];
#pragma unroll
        for (int ii = 0; ii < N; ++ii) {
            const float h = __ldg(Hpost + t * N + ii);
            hp2[ii] = f2_make(h, h);
        }
        // n = 8: the dH_res sums are scalars, each chunk's four channel pairs
        // folded into them (as pairs they take 128 registers and the kernel
        // spills)
        constexpr bool SR1 = N == 8;
        f32x2 sR[SR1 ? 1 : N * N], sP[N], sQ[N];
        float sR1[SR1 ? N * N : 1];
#pragma unroll
        for (int e = 0; e < (SR1 ? 1 : N * N); ++e) sR[e] = 0ull;
#pragma unroll
        for (int e = 0; e < (SR1 ? N * N : 1); ++e) sR1[e] = 0.f;
#pragma unroll
        for (int j = 0; j < N; ++j) sP[j] = sQ[j] = 0ull;

        for (int64_t base = lane; base < C8; base += 32 * U) {
            uint4 dr[U][N], xr[U][N], fv[U], yv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c8 = base + 32 * u;
                if (U == 1 || c8 < C8) {
#pragma unroll
                    for (int ii = 0; ii < N; ++ii)
                        dr[u][ii] = ld_stream(dout + ((t * N + ii) * C8 + c8) * 8);
#pragma unroll
                    for (int j = 0; j < N; ++j) xr[u][j] = ld_stream(x + ((t * N + j) * C8 + c8) * 8);
                    fv[u] = ld_stream(f + (t * C8 + c8) * 8);
                    yv[u] = ld_stream(dy + (t * C8 + c8) * 8);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c8 = base + 32 * u;
                if (U > 1 && c8 >= C8) continue;
                f32x2 fb[4], gy[4];
                unpack8x2(fv[u], fb);
                unpack8x2(yv[u], gy);
                if (bias) {
                    f32x2 bv[4];
                    unpack8x2(__ldg(reinterpret_cast<const uint4 *>(bias + c8 * 8)), bv);
#pragma unroll
                    for (int p = 0; p < 4; ++p) fb[p] = f2_add(fb[p], bv[p]);
                }
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    f32x2 v[4];
                    unpack8x2(xr[u][j], v);
#pragma unroll
                    for (int p = 0; p < 4; ++p) sQ[j] = f2_fma(gy[p], v[p], sQ[j]);
                }
                f32x2 dfv[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int ii = 0; ii < N; ++ii) {
                    f32x2 d[4];
                    unpack8x2(dr[u][ii], d);
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        sP[ii] = f2_fma(d[p], fb[p], sP[ii]);
                        dfv[p] = f2_fma(hp2[ii], d[p], dfv[p]);
                    }
#pragma unroll
                    for (int j = 0; j < N; ++j) {
                        f32x2 v[4];
                        unpack8x2(xr[u][j], v);
                        if (SR1) {
                            f32x2 c = f2_mul(v[0], d[0]);
#pragma unroll
                            for (int p = 1; p < 4; ++p) c = f2_fma(v[p], d[p], c);
                            float lo, hi;
                            f2_split(c, lo, hi);
                            sR1[j * N + ii] += lo + hi;
                        } else {
#pragma unroll
                            for (int p = 0; p < 4; ++p)
                                sR[j * N + ii] = f2_fma(v[p], d[p], sR[j * N + ii]);
                        }
                    }
                }
                if (df) st_stream(df + (t * C8 + c8) * 8, pack8x2(dfv));
            }
        }
        float aR[N * N], aP[N], aQ[N];
        auto fold = [](f32x2 v) {
            float lo, hi;
            f2_split(v, lo, hi);
            return lo + hi;
        };
#pragma unroll
        for (int e = 0; e < N * N; ++e) aR[e] = SR1 ? sR1[e] : fold(sR[SR1 ? 0 : e]);
#pragma unroll
        for (int j = 0; j < N; ++j) {
            aP[j] = fold(sP[j]);
            aQ[j] = fold(sQ[j]);
        }
#pragma unroll
        for (int e = 0; e < N * N; ++e) aR[e] = warp_sum(aR[e]);
#pragma unroll
        for (int j = 0; j < N; ++j) {
            aP[j] = warp_sum(aP[j]);
            aQ[j] = warp_sum(aQ[j]);
        }
        if (lane == 0) {
            float4 *r4 = reinterpret_cast<float4 *>(dHres + t * N * N);
#pragma unroll
            for (int e = 0; e < N * N; e += 4)
                r4[e / 4] = make_float4(aR[e], aR[e + 1], aR[e + 2], aR[e + 3]);
            float4 *p4 = reinterpret_cast<float4 *>(dHpost + t * N);
            float4 *q4 = reinterpret_cast<float4 *>(dHpre + t * N);
#pragma unroll
            for (int j = 0; j < N; j += 4) {
                p4[j / 4] = make_float4(aP[j], aP[j + 1], aP[j + 2], aP[j + 3]);
                q4[j / 4] = make_float4(aQ[j], aQ[j + 1], aQ[j + 2], aQ[j + 3]);
            }
        }
    }
}

int bwd_tok_blocks(int64_t T)
{
    const int64_t want = (T + kTokWarps - 1) / kTokWarps;
    const int64_t cap = int64_t(kSplitSms) * 2;
    return int(want < cap ? (want > 0 ? want : 1) : cap);
}

cudaError_t launch_bwd_tok(const bf16 *dout, const bf16 *x, const bf16 *f, const bf16 *bias,
                           const bf16 *dy, const float *Hpost, int64_t T, int n, int64_t C,
                           bf16 *df, float *dHres, float *dHpost, float *dHpre, cudaStream_t s)
{
    const unsigned g = unsigned(bwd_tok_blocks(T));
    MHC_PROF("k_bwd_tok", s);
    if (n == 4)
        launch_k(k_bwd_tok<4, MHC_TOK_U>, dim3(g), dim3(32 * kTokWarps), 0, s, dout, x, f, bias, dy, Hpost, T, C / 8,
                                                             df, dHres, dHpost, dHpre);
    else
        launch_k(k_bwd_tok<8, 1>, dim3(g), dim3(32 * kTokWarps), 0, s, dout, x, f, bias, dy, Hpost, T, C / 8, df,
                                                     dHres, dHpost, dHpre);
    return cudaGetLastError();
}

}  // namespace mhc
