// Token pass of the mHC layer backward: one read of dout, x, f and dy.
//
// One warp per token streams the token's rows once and forms
//   dH_res[j][i] = sum_c x[j][c] dout[i][c]      dH_post[i] = sum_c dout[i][c] (f[c] + bias[c])
//   dH_pre[i]    = sum_c dy[c] x[i][c]           df[c]      = sum_i H_post[i] dout[i][c]
// (Megatron-Core fused_mhc_kernels _torch_h_post_bda_bwd and
// _torch_h_aggregate_bwd), then takes the token through the compute_h
// backward on the same warp (gate derivatives, Sinkhorn backward, RMS scale:
// rwkv-ops mhu_ffi.cu MhcPreOpBwdHost, RL-Kernel PR #383 fp32_gemm_rms) and
// writes what the residual-gradient pass reads: du = alpha_seg r dz as bf16
// hi | lo, H_post as bf16 hi | lo, and coef = -dr r^2 / (K q).
//
// The sums over tokens of dz (db) and of the three dalpha terms are kept per
// warp in token order, then summed per block in warp order into one partial
// row per block; k_bwd_finalize adds the rows in block order.
#include "launch.h"
#include "sinkhorn.cuh"

namespace mhc {

constexpr int kTokWarps = 8;

template <int N>
__global__ void __launch_bounds__(256)
    k_bwd_tok(const bf16 *__restrict__ dout, const bf16 *__restrict__ x,
              const bf16 *__restrict__ f, const bf16 *__restrict__ bias,
              const bf16 *__restrict__ dy, const float *__restrict__ Hpost,
              const float *__restrict__ u_save, const float *__restrict__ r_save,
              const float *__restrict__ alpha, const float *__restrict__ b, int64_t T,
              int64_t C8, int iters, float eps_sk, float eps_rms, bf16 *__restrict__ df,
              bf16 *__restrict__ du_hl, int du_cols, float *__restrict__ coef,
              float *__restrict__ part)
{
    constexpr int O = N * N + 2 * N;
    constexpr int PW = O + 4;  // partial row: dz sums [0,O), dalpha terms [O,O+3), pad
    extern __shared__ float sm[];  // [warps][2*iters][N] Sinkhorn denominators, then [warps][PW]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int i = lane & (N - 1);
    // every lane group of the warp runs the token's Sinkhorn on identical
    // values, so the groups share one copy of the stored denominators
    float *store = sm + warp * (2 * iters * N) + i;
    const float Kf = float(int64_t(N) * C8 * 8);
    const float a0 = __ldg(alpha), a1 = __ldg(alpha + 1), a2 = __ldg(alpha + 2);
    float zpre_acc = 0.f, zpost_acc = 0.f, zres_acc[N], ga_acc[3] = {0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < N; ++j) zres_acc[j] = 0.f;

    const int64_t warps = int64_t(gridDim.x) * kTokWarps;
    for (int64_t t = int64_t(blockIdx.x) * kTokWarps + warp; t < T; t += warps) {
        float hp[N];
#pragma unroll
        for (int ii = 0; ii < N; ++ii) hp[ii] = __ldg(Hpost + t * N + ii);
        float aR[N * N], aP[N], aQ[N];
#pragma unroll
        for (int e = 0; e < N * N; ++e) aR[e] = 0.f;
#pragma unroll
        for (int j = 0; j < N; ++j) aP[j] = aQ[j] = 0.f;

        for (int64_t c8 = lane; c8 < C8; c8 += 32) {
            uint4 dr[N], xr[N];
#pragma unroll
            for (int ii = 0; ii < N; ++ii) dr[ii] = ld_stream(dout + ((t * N + ii) * C8 + c8) * 8);
#pragma unroll
            for (int j = 0; j < N; ++j) xr[j] = ld_stream(x + ((t * N + j) * C8 + c8) * 8);
            float fb[8], gy[8];
            unpack8(ld_stream(f + (t * C8 + c8) * 8), fb);
            unpack8(ld_stream(dy + (t * C8 + c8) * 8), gy);
            if (bias) {
                float bv[8];
                unpack8(__ldg(reinterpret_cast<const uint4 *>(bias + c8 * 8)), bv);
#pragma unroll
                for (int e = 0; e < 8; ++e) fb[e] += bv[e];
            }
#pragma unroll
            for (int j = 0; j < N; ++j) {
                float v[8];
                unpack8(xr[j], v);
                float s = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) s = fmaf(gy[e], v[e], s);
                aQ[j] += s;
            }
            float dfv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ii = 0; ii < N; ++ii) {
                float d[8];
                unpack8(dr[ii], d);
                float sp = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    sp = fmaf(d[e], fb[e], sp);
                    dfv[e] = fmaf(hp[ii], d[e], dfv[e]);
                }
                aP[ii] += sp;
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    float v[8];
                    unpack8(xr[j], v);
                    float s = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) s = fmaf(v[e], d[e], s);
                    aR[j * N + ii] += s;
                }
            }
            if (df) st_stream(df + (t * C8 + c8) * 8, pack8(dfv));
        }
#pragma unroll
        for (int e = 0; e < N * N; ++e) aR[e] = warp_sum(aR[e]);
#pragma unroll
        for (int j = 0; j < N; ++j) {
            aP[j] = warp_sum(aP[j]);
            aQ[j] = warp_sum(aQ[j]);
        }

        // compute_h backward of token t; lane i of each group owns row i
        float g[N], dhpre = 0.f, dhpost = 0.f, hpi = 0.f;
#pragma unroll
        for (int ii = 0; ii < N; ++ii)
            if (ii == i) {
#pragma unroll
                for (int j = 0; j < N; ++j) g[j] = aR[ii * N + j];  // dL/dH_res[i][j]
                dhpre = aQ[ii];
                dhpost = aP[ii];
                hpi = hp[ii];
            }
        const float *u = u_save + t * O;
        const float r = __ldg(r_save + t);
        const float upre = __ldg(u + i), upost = __ldg(u + N + i);
        float ures[N], e[N], a[N];
#pragma unroll
        for (int j = 0; j < N; ++j) {
            ures[j] = __ldg(u + 2 * N + i * N + j);
            e[j] = expf(a2 * r * ures[j] + __ldg(b + 2 * N + i * N + j));
            a[j] = e[j];
        }
        sk_forward<N>(a, iters, eps_sk, store, N);
        sk_backward<N>(g, a, e, iters, store, N);  // g = dz_res row i
        const float sp = sigmoidf_(a0 * r * upre + __ldg(b + i));
        const float so = sigmoidf_(a1 * r * upost + __ldg(b + N + i));
        const float dzpre = dhpre * sp * (1.f - sp);
        const float dzpost = dhpost * 2.f * so * (1.f - so);
        float gres = 0.f;
#pragma unroll
        for (int j = 0; j < N; ++j) gres = fmaf(g[j], ures[j], gres);
        float gpre = dzpre * upre, gpost = dzpost * upost;
#pragma unroll
        for (int m = 1; m < N; m <<= 1) {
            gpre += __shfl_xor_sync(kFull, gpre, m);
            gpost += __shfl_xor_sync(kFull, gpost, m);
            gres += __shfl_xor_sync(kFull, gres, m);
        }
        bf16 *dut = du_hl + t * du_cols;
        if (lane < N) {
            auto put = [&](int o, float v) {
                const bf16 hi = __float2bfloat16_rn(v);
                dut[o] = hi;
                dut[O + o] = __float2bfloat16_rn(v - __bfloat162float(hi));
            };
            put(i, a0 * r * dzpre);
            put(N + i, a1 * r * dzpost);
#pragma unroll
            for (int j = 0; j < N; ++j) put(2 * N + i * N + j, a2 * r * g[j]);
            const bf16 hph = __float2bfloat16_rn(hpi);
            dut[2 * O + i] = hph;
            dut[2 * O + N + i] = __float2bfloat16_rn(hpi - __bfloat162float(hph));
        }
        for (int o = 2 * O + 2 * N + lane; o < du_cols; o += 32) dut[o] = __float2bfloat16_rn(0.f);
        if (lane == 0) {
            const float dr = a0 * gpre + a1 * gpost + a2 * gres;
            const float q = 1.0f / r - eps_rms;
            coef[t] = (q > 0.f) ? -dr * r * r / (Kf * q) : 0.f;
        }
        zpre_acc += dzpre;
        zpost_acc += dzpost;
#pragma unroll
        for (int j = 0; j < N; ++j) zres_acc[j] += g[j];
        ga_acc[0] += gpre * r;
        ga_acc[1] += gpost * r;
        ga_acc[2] += gres * r;
        __syncwarp();
    }

    float *red = sm + kTokWarps * 2 * iters * N;
    if (lane < N) {
        red[warp * PW + i] = zpre_acc;
        red[warp * PW + N + i] = zpost_acc;
#pragma unroll
        for (int j = 0; j < N; ++j) red[warp * PW + 2 * N + i * N + j] = zres_acc[j];
    }
    if (lane == 0) {
        red[warp * PW + O] = ga_acc[0];
        red[warp * PW + O + 1] = ga_acc[1];
        red[warp * PW + O + 2] = ga_acc[2];
        red[warp * PW + O + 3] = 0.f;
    }
    __syncthreads();
    if (threadIdx.x < PW) {
        float s = 0.f;
        for (int w = 0; w < kTokWarps; ++w) s += red[w * PW + threadIdx.x];
        part[int64_t(blockIdx.x) * PW + threadIdx.x] = s;
    }
}

int bwd_tok_blocks(int64_t T)
{
    const int64_t want = (T + kTokWarps - 1) / kTokWarps;
    const int64_t cap = int64_t(kSplitSms) * 8;
    return int(want < cap ? (want > 0 ? want : 1) : cap);
}

cudaError_t launch_bwd_tok(const bf16 *dout, const bf16 *x, const bf16 *f, const bf16 *bias,
                           const bf16 *dy, const float *Hpost, const float *u_save,
                           const float *r_save, const float *alpha, const float *b, int64_t T,
                           int n, int64_t C, int iters, float eps_sk, float eps_rms, bf16 *df,
                           bf16 *du_hl, int du_cols, float *coef, float *part, cudaStream_t s)
{
    const unsigned g = unsigned(bwd_tok_blocks(T));
    const size_t smem = size_t(kTokWarps) * (2 * iters * n + bwd_part_cols(n)) * sizeof(float);
    MHC_PROF("k_bwd_tok", s);
    if (n == 4)
        k_bwd_tok<4><<<g, 32 * kTokWarps, smem, s>>>(dout, x, f, bias, dy, Hpost, u_save, r_save,
                                                     alpha, b, T, C / 8, iters, eps_sk, eps_rms,
                                                     df, du_hl, du_cols, coef, part);
    else
        k_bwd_tok<8><<<g, 32 * kTokWarps, smem, s>>>(dout, x, f, bias, dy, Hpost, u_save, r_save,
                                                     alpha, b, T, C / 8, iters, eps_sk, eps_rms,
                                                     df, du_hl, du_cols, coef, part);
    return cudaGetLastError();
}

}  // namespace mhc
