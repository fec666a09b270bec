// proj_rms_compute_h forward and backward, and the layer backward's
// residual-gradient pass.
//
// Definitions: Megatron-Core fused_mhc_kernels (fused_proj_rms_compute_h,
// _torch_proj_rms_compute_h(x, weight, alpha_pre, alpha_post, alpha_res,
// bias, n, eps, compute_h_eps)), RL-Kernel PR #383 (fp32_gemm_rms: r =
// 1/(q + eps), q = sqrt(s/K), backward term -r^2 x/(K q) guarded at an
// all-zero row; three alpha scalars over PRE/POST/COMB), rwkv-ops mhu_ffi.cu
// (MhcPreOpFwdHost: H_pre after sigmoid, H_post after 2*sigmoid, H_res after
// Sinkhorn; MhcPreOpBwdHost: gradient back to the raw logits).
//
// Forward:  k_proj_tc (k_proj_tc.cu: split-K partial u = x W and s = sum x^2
//           on the tensor cores), k_compute_h_fwd (sum of partials, r, z,
//           gates, Sinkhorn)
// Backward: [layer: k_bwd_tok (k_bwd_tok.cu), the per-token dH sums and df]
//           k_compute_h_bwd (per-token du as bf16 hi|lo, RMS coefficient,
//           per-block sums of dz and the dalpha terms), k_bwd_tc (k_bwd_tc.cu: du W^T + coef x [+ H_res dout + H_pre dy],
//           dW and dbias on the tensor cores) and k_bwd_finalize, the
//           fixed-order sums for db, dalpha (and dW, dbias when split).
#include "launch.h"
#include "sinkhorn.cuh"

namespace mhc {

template <int N>
struct Dims {
    static constexpr int O = N * N + 2 * N;
    static constexpr int OP = (O + 7) / 8;  // logits per thread in the GEMM (o = og + 8p)
};

// ---------------------------------------------------------------------------
// compute_h forward.  A group of N lanes per token, lane i owns row i of the
// n x n block and logits pre[i], post[i], res[i][0..N).
// ---------------------------------------------------------------------------
template <int N>
__global__ void __launch_bounds__(128)
    k_compute_h_fwd(const float *__restrict__ upart, const float *__restrict__ spart, int splits,
                    const float *__restrict__ alpha, const float *__restrict__ b, int64_t T,
                    int64_t K, int iters, float eps_sk, float eps_rms, float *__restrict__ Hpre,
                    float *__restrict__ Hpost, float *__restrict__ Hres,
                    float *__restrict__ u_save, float *__restrict__ r_save)
{
    pdl_wait();
    constexpr int O = Dims<N>::O;
    const int64_t gt = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t t = gt / N;
    const int i = int(gt % N);
    const bool live = t < T;
    const int64_t tt = live ? t : 0;
    float s = 0.f, upre = 0.f, upost = 0.f, ures[N];
#pragma unroll
    for (int j = 0; j < N; ++j) ures[j] = 0.f;
    for (int sp = 0; sp < splits; ++sp) {
        const float *u = upart + (int64_t(sp) * T + tt) * O;
        s += __ldg(spart + int64_t(sp) * T + tt);
        upre += __ldg(u + i);
        upost += __ldg(u + N + i);
#pragma unroll
        for (int j = 0; j < N; ++j) ures[j] += __ldg(u + 2 * N + i * N + j);
    }
    const float q = sqrtf(s / float(K));
    const float r = 1.0f / (q + eps_rms);
    const float a0 = __ldg(alpha), a1 = __ldg(alpha + 1), a2 = __ldg(alpha + 2);
    const float zpre = a0 * r * upre + __ldg(b + i);
    const float zpost = a1 * r * upost + __ldg(b + N + i);
    float a[N];
#pragma unroll
    for (int j = 0; j < N; ++j) a[j] = expf(a2 * r * ures[j] + __ldg(b + 2 * N + i * N + j));
    sk_forward<N>(a, iters, eps_sk, nullptr, 0);
    if (live) {
        Hpre[t * N + i] = sigmoidf_(zpre);
        Hpost[t * N + i] = 2.0f * sigmoidf_(zpost);
#pragma unroll
        for (int j = 0; j < N; ++j) Hres[(t * N + i) * N + j] = a[j];
        if (u_save) {
            u_save[t * O + i] = upre;
            u_save[t * O + N + i] = upost;
#pragma unroll
            for (int j = 0; j < N; ++j) u_save[t * O + 2 * N + i * N + j] = ures[j];
        }
        if (r_save && i == 0) r_save[t] = r;
    }
}

// ---------------------------------------------------------------------------
// compute_h backward.  Same lane layout.  Per token writes
//   du[t][o] = alpha_seg r dz[o] (bf16 hi | lo; fp32 when du_f32 is given),
//   dub[t] = sum_o |du[t][o]| (when given: the residual-gradient pass bounds
//   the error of its bf16 product with it) and
//   coef[t] = -dr r^2 / (K q) with dr = sum_o dz alpha_seg u and q = 1/r - eps_rms
//   (coef = 0 when q <= 0: an all-zero row has zero RMS gradient);
// per block one partial row: the block's sums of dz[o] (in token order) and
// of the dalpha terms ga[seg] = sum_{o in seg} dz r u.
// ---------------------------------------------------------------------------
template <int N>
__global__ void __launch_bounds__(128)
    k_compute_h_bwd(const float *__restrict__ dHpre, const float *__restrict__ dHpost,
                    const float *__restrict__ dHres, const float *__restrict__ u_save,
                    const float *__restrict__ r_save, const float *__restrict__ alpha,
                    const float *__restrict__ b, int64_t T, int64_t K, int iters, float eps_sk,
                    float eps_rms, bf16 *__restrict__ du_hl, int du_cols,
                    float *__restrict__ coef, float *__restrict__ part,
                    const float *__restrict__ s_tot, float *__restrict__ du_f32,
                    float *__restrict__ dub, const float *__restrict__ Hres,
                    float *__restrict__ HresT)
{
    pdl_wait();
    constexpr int O = Dims<N>::O;
    constexpr int PW = O + 4, TB = 128 / N;
    extern __shared__ float sk_store[];  // [2*iters][blockDim.x]
    if (HresT) {
        // the layer's H_res transposed, HresT[t][i][j] = H_res[t][j][i], for
        // the residual-gradient pass (lane i of a token copies row i of
        // H_res into column i)
        const int64_t gt0 = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
        const int64_t t0 = gt0 / N;
        const int i0 = int(gt0 % N);
        if (t0 < T) {
#pragma unroll
            for (int j = 0; j < N; ++j) HresT[(t0 * N + j) * N + i0] = __ldg(Hres + (t0 * N + i0) * N + j);
        }
    }
    __shared__ float red[TB][PW];
    const int64_t gt = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t t = gt / N;
    const int i = int(gt % N);
    const int tb = threadIdx.x / N;
    const bool live = t < T;
    const int64_t tt = live ? t : 0;
    const float *u = u_save + tt * O;
    // r from the forward, or from the summed squares of a sharded forward
    const float r = r_save ? __ldg(r_save + tt)
                           : 1.0f / (sqrtf(__ldg(s_tot + tt) / float(K)) + eps_rms);
    const float a0 = __ldg(alpha), a1 = __ldg(alpha + 1), a2 = __ldg(alpha + 2);
    const float upre = __ldg(u + i), upost = __ldg(u + N + i);
    const float zpre = a0 * r * upre + __ldg(b + i);
    const float zpost = a1 * r * upost + __ldg(b + N + i);
    float ures[N], e[N], a[N], g[N];
#pragma unroll
    for (int j = 0; j < N; ++j) {
        ures[j] = __ldg(u + 2 * N + i * N + j);
        e[j] = expf(a2 * r * ures[j] + __ldg(b + 2 * N + i * N + j));
        a[j] = e[j];
        g[j] = live ? __ldg(dHres + (tt * N + i) * N + j) : 0.f;
    }
    float *store = sk_store + threadIdx.x;
    sk_forward<N>(a, iters, eps_sk, store, blockDim.x);
    sk_backward<N>(g, a, e, iters, store, blockDim.x);  // g = dz_res row i
    const float sp = sigmoidf_(zpre), so = sigmoidf_(zpost);
    const float dzpre = (live ? __ldg(dHpre + tt * N + i) : 0.f) * sp * (1.f - sp);
    const float dzpost = (live ? __ldg(dHpost + tt * N + i) : 0.f) * 2.f * so * (1.f - so);
    float gres = 0.f;
#pragma unroll
    for (int j = 0; j < N; ++j) gres = fmaf(g[j], ures[j], gres);
    float gpre = dzpre * upre, gpost = dzpost * upost;
    // this lane's du terms and the sum of their magnitudes
    const float dupre = a0 * r * dzpre, dupost = a1 * r * dzpost;
    float dures[N];
    float sabs = fabsf(dupre) + fabsf(dupost);
#pragma unroll
    for (int j = 0; j < N; ++j) {
        dures[j] = a2 * r * g[j];
        sabs += fabsf(dures[j]);
    }
    // sums over the N lanes of the group
#pragma unroll
    for (int m = 1; m < N; m <<= 1) {
        gpre += __shfl_xor_sync(kFull, gpre, m);
        gpost += __shfl_xor_sync(kFull, gpost, m);
        gres += __shfl_xor_sync(kFull, gres, m);
        sabs += __shfl_xor_sync(kFull, sabs, m);
    }
    if (live) {
        // du = alpha_seg r dz, stored as bf16 hi (columns [0,O)) and the bf16
        // remainder (columns [O,2O)); zero columns pad the row to du_cols.
        bf16 *dut = du_hl + t * du_cols;
        auto put = [&](int o, float v) {
            const bf16 hi = __float2bfloat16_rn(v);
            dut[o] = hi;
            dut[O + o] = __float2bfloat16_rn(v - __bfloat162float(hi));
            if (du_f32) du_f32[t * O + o] = v;
        };
        put(i, dupre);
        put(N + i, dupost);
#pragma unroll
        for (int j = 0; j < N; ++j) put(2 * N + i * N + j, dures[j]);
        // columns [2O, 2O+2N): H_post[i] as bf16 hi | lo (the dbias MMA of the
        // residual-gradient pass reads them), then zeros
        const float hp = 2.0f * so;
        const bf16 hph = __float2bfloat16_rn(hp);
        dut[2 * O + i] = hph;
        dut[2 * O + N + i] = __float2bfloat16_rn(hp - __bfloat162float(hph));
        if (i == 0) {
            for (int o = 2 * O + 2 * N; o < du_cols; ++o) dut[o] = __float2bfloat16_rn(0.f);
            const float dr = a0 * gpre + a1 * gpost + a2 * gres;
            const float q = 1.0f / r - eps_rms;
            coef[t] = (q > 0.f) ? -dr * r * r / (float(K) * q) : 0.f;
            if (dub) dub[t] = sabs;
        }
    }
    // this token's row of the block partial (zeros for a dead token)
    red[tb][i] = live ? dzpre : 0.f;
    red[tb][N + i] = live ? dzpost : 0.f;
#pragma unroll
    for (int j = 0; j < N; ++j) red[tb][2 * N + i * N + j] = live ? g[j] : 0.f;
    if (i == 0) {
        red[tb][O] = live ? gpre * r : 0.f;
        red[tb][O + 1] = live ? gpost * r : 0.f;
        red[tb][O + 2] = live ? gres * r : 0.f;
        red[tb][O + 3] = 0.f;
    }
    __syncthreads();
    if (threadIdx.x < PW) {
        float acc = 0.f;
        for (int k = 0; k < TB; ++k) acc += red[k][threadIdx.x];
        part[int64_t(blockIdx.x) * PW + threadIdx.x] = acc;
    }
}

// ---------------------------------------------------------------------------
// n = 4: one thread per token, the 4 x 4 Sinkhorn in its registers
// (sk4_forward / sk4_backward).  The same formulas as above; the n lanes'
// butterfly sums become (v0 + v1) + (v2 + v3) over the rows.  The backward
// keeps 32 tokens per block, so its partial rows are those of the lane form.
// ---------------------------------------------------------------------------
constexpr int kCh4Fwd = 64;

__global__ void __launch_bounds__(kCh4Fwd)
    k_compute_h_fwd4(const float *__restrict__ upart, const float *__restrict__ spart, int splits,
                     const float *__restrict__ alpha, const float *__restrict__ b, int64_t T,
                     int64_t K, int iters, float eps_sk, float eps_rms, float *__restrict__ Hpre,
                     float *__restrict__ Hpost, float *__restrict__ Hres,
                     float *__restrict__ u_save, float *__restrict__ r_save)
{
    pdl_wait();
    constexpr int N = 4, O = Dims<4>::O;
    const int64_t t = int64_t(blockIdx.x) * kCh4Fwd + threadIdx.x;
    if (t >= T) return;
    float u[O], s = 0.f;
#pragma unroll
    for (int o = 0; o < O; ++o) u[o] = 0.f;
    for (int sp = 0; sp < splits; ++sp) {
        s += __ldg(spart + int64_t(sp) * T + t);
        const float4 *up = reinterpret_cast<const float4 *>(upart + (int64_t(sp) * T + t) * O);
#pragma unroll
        for (int q4 = 0; q4 < O / 4; ++q4) {
            const float4 v = __ldg(up + q4);
            u[4 * q4] += v.x;
            u[4 * q4 + 1] += v.y;
            u[4 * q4 + 2] += v.z;
            u[4 * q4 + 3] += v.w;
        }
    }
    const float q = sqrtf(s / float(K));
    const float r = 1.0f / (q + eps_rms);
    const float a0 = __ldg(alpha), a1 = __ldg(alpha + 1), a2 = __ldg(alpha + 2);
    float hp[N], hq[N], a[N][N];
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float zpre = a0 * r * u[i] + __ldg(b + i);
        const float zpost = a1 * r * u[N + i] + __ldg(b + N + i);
        hp[i] = sigmoidf_(zpre);
        hq[i] = 2.0f * sigmoidf_(zpost);
#pragma unroll
        for (int j = 0; j < N; ++j)
            a[i][j] = expf(a2 * r * u[2 * N + i * N + j] + __ldg(b + 2 * N + i * N + j));
    }
    sk4_forward(a, iters, eps_sk, nullptr, 0);
    reinterpret_cast<float4 *>(Hpre)[t] = make_float4(hp[0], hp[1], hp[2], hp[3]);
    reinterpret_cast<float4 *>(Hpost)[t] = make_float4(hq[0], hq[1], hq[2], hq[3]);
#pragma unroll
    for (int i = 0; i < N; ++i)
        reinterpret_cast<float4 *>(Hres)[t * N + i] = make_float4(a[i][0], a[i][1], a[i][2], a[i][3]);
    if (u_save) {
        float4 *us = reinterpret_cast<float4 *>(u_save + t * O);
#pragma unroll
        for (int q4 = 0; q4 < O / 4; ++q4)
            us[q4] = make_float4(u[4 * q4], u[4 * q4 + 1], u[4 * q4 + 2], u[4 * q4 + 3]);
    }
    if (r_save) r_save[t] = r;
}

constexpr int kCh4Bwd = 32;
constexpr int kCh4DuCols = 64;   // du_hl columns at n = 4

__global__ void __launch_bounds__(kCh4Bwd)
    k_compute_h_bwd4(const float *__restrict__ dHpre, const float *__restrict__ dHpost,
                     const float *__restrict__ dHres, const float *__restrict__ u_save,
                     const float *__restrict__ r_save, const float *__restrict__ alpha,
                     const float *__restrict__ b, int64_t T, int64_t K, int iters, float eps_sk,
                     float eps_rms, bf16 *__restrict__ du_hl, float *__restrict__ coef,
                     float *__restrict__ part, const float *__restrict__ s_tot,
                     float *__restrict__ du_f32, float *__restrict__ dub)
{
    pdl_wait();
    constexpr int N = 4, O = Dims<4>::O, PW = O + 4;
    extern __shared__ float sk_store[];   // [8 iters][kCh4Bwd]
    __shared__ float red[kCh4Bwd][PW + 1];
    const int tid = threadIdx.x;
    const int64_t t = int64_t(blockIdx.x) * kCh4Bwd + tid;
    const bool live = t < T;
    const int64_t tt = live ? t : 0;
    float u[O];
#pragma unroll
    for (int q4 = 0; q4 < O / 4; ++q4) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(u_save + tt * O) + q4);
        u[4 * q4] = v.x;
        u[4 * q4 + 1] = v.y;
        u[4 * q4 + 2] = v.z;
        u[4 * q4 + 3] = v.w;
    }
    // r from the forward, or from the summed squares of a sharded forward
    const float r = r_save ? __ldg(r_save + tt)
                           : 1.0f / (sqrtf(__ldg(s_tot + tt) / float(K)) + eps_rms);
    const float a0 = __ldg(alpha), a1 = __ldg(alpha + 1), a2 = __ldg(alpha + 2);
    float e[N][N], a[N][N], g[N][N];
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float4 gv = live ? __ldg(reinterpret_cast<const float4 *>(dHres + tt * N * N) + i)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        g[i][0] = gv.x;
        g[i][1] = gv.y;
        g[i][2] = gv.z;
        g[i][3] = gv.w;
#pragma unroll
        for (int j = 0; j < N; ++j) {
            e[i][j] = expf(a2 * r * u[2 * N + i * N + j] + __ldg(b + 2 * N + i * N + j));
            a[i][j] = e[i][j];
        }
    }
    float *store = sk_store + tid;
    sk4_forward(a, iters, eps_sk, store, kCh4Bwd);
    sk4_backward(g, a, e, iters, store, kCh4Bwd);   // g = dz_res
    const float4 dhp = live ? __ldg(reinterpret_cast<const float4 *>(dHpre) + tt) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float4 dhq = live ? __ldg(reinterpret_cast<const float4 *>(dHpost) + tt) : make_float4(0.f, 0.f, 0.f, 0.f);
    const float dhpv[N] = {dhp.x, dhp.y, dhp.z, dhp.w}, dhqv[N] = {dhq.x, dhq.y, dhq.z, dhq.w};
    float dzpre[N], dzpost[N], hq[N], gr[N], pr[N], po[N], sb[N];
    float dv[O];   // du in column order
#pragma unroll
    for (int i = 0; i < N; ++i) {
        const float sp = sigmoidf_(a0 * r * u[i] + __ldg(b + i));
        const float so = sigmoidf_(a1 * r * u[N + i] + __ldg(b + N + i));
        hq[i] = 2.0f * so;
        dzpre[i] = dhpv[i] * sp * (1.f - sp);
        dzpost[i] = dhqv[i] * 2.f * so * (1.f - so);
        pr[i] = dzpre[i] * u[i];
        po[i] = dzpost[i] * u[N + i];
        float gi = 0.f;
#pragma unroll
        for (int j = 0; j < N; ++j) gi = fmaf(g[i][j], u[2 * N + i * N + j], gi);
        gr[i] = gi;
        dv[i] = a0 * r * dzpre[i];
        dv[N + i] = a1 * r * dzpost[i];
        float sa = fabsf(dv[i]) + fabsf(dv[N + i]);
#pragma unroll
        for (int j = 0; j < N; ++j) {
            dv[2 * N + i * N + j] = a2 * r * g[i][j];
            sa += fabsf(dv[2 * N + i * N + j]);
        }
        sb[i] = sa;
    }
    const float gpre = (pr[0] + pr[1]) + (pr[2] + pr[3]);
    const float gpost = (po[0] + po[1]) + (po[2] + po[3]);
    const float gres = (gr[0] + gr[1]) + (gr[2] + gr[3]);
    const float sabs = (sb[0] + sb[1]) + (sb[2] + sb[3]);
    if (live) {
        // du_hl row: bf16(du) in columns [0, O), the bf16 remainder in
        // [O, 2O), H_post as bf16 hi | lo in [2O, 2O + 2n), zeros to 64
        auto col = [&](int c) -> float {
            if (c < O) return __bfloat162float(__float2bfloat16_rn(dv[c]));
            if (c < 2 * O) {
                const float v = dv[c - O];
                return v - __bfloat162float(__float2bfloat16_rn(v));
            }
            if (c < 2 * O + N) return hq[c - 2 * O];
            if (c < 2 * O + 2 * N) {
                const float v = hq[c - 2 * O - N];
                return v - __bfloat162float(__float2bfloat16_rn(v));
            }
            return 0.f;
        };
        uint4 *row = reinterpret_cast<uint4 *>(du_hl + t * kCh4DuCols);
#pragma unroll
        for (int c8 = 0; c8 < kCh4DuCols / 8; ++c8) {
            float v8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v8[k] = col(8 * c8 + k);
            row[c8] = pack8(v8);
        }
        if (du_f32) {
            float4 *d4 = reinterpret_cast<float4 *>(du_f32 + t * O);
#pragma unroll
            for (int q4 = 0; q4 < O / 4; ++q4)
                d4[q4] = make_float4(dv[4 * q4], dv[4 * q4 + 1], dv[4 * q4 + 2], dv[4 * q4 + 3]);
        }
        const float dr = a0 * gpre + a1 * gpost + a2 * gres;
        const float q = 1.0f / r - eps_rms;
        coef[t] = (q > 0.f) ? -dr * r * r / (float(K) * q) : 0.f;
        if (dub) dub[t] = sabs;
    }
    // this token's row of the block partial (zeros for a dead token)
#pragma unroll
    for (int i = 0; i < N; ++i) {
        red[tid][i] = live ? dzpre[i] : 0.f;
        red[tid][N + i] = live ? dzpost[i] : 0.f;
#pragma unroll
        for (int j = 0; j < N; ++j) red[tid][2 * N + i * N + j] = live ? g[i][j] : 0.f;
    }
    red[tid][O] = live ? gpre * r : 0.f;
    red[tid][O + 1] = live ? gpost * r : 0.f;
    red[tid][O + 2] = live ? gres * r : 0.f;
    red[tid][O + 3] = 0.f;
    __syncwarp();
    if (tid < PW) {
        float acc = 0.f;
        for (int k = 0; k < kCh4Bwd; ++k) acc += red[k][tid];
        part[int64_t(blockIdx.x) * PW + tid] = acc;
    }
}

// The compute_h forward launch (lane form for n = 8)
template <int N>
static void launch_ch_fwd(const float *upart, const float *spart, int S, const float *alpha,
                          const float *b, int64_t T, int64_t K, int iters, float eps_sk,
                          float eps_rms, float *Hpre, float *Hpost, float *Hres, float *u_save,
                          float *r_save, cudaStream_t s)
{
    MHC_PROF("k_compute_h_fwd", s);
    if constexpr (N == 4)
        launch_k(k_compute_h_fwd4, dim3(unsigned((T + kCh4Fwd - 1) / kCh4Fwd)), dim3(kCh4Fwd), 0, s,
                 upart, spart, S, alpha, b, T, K, iters, eps_sk, eps_rms, Hpre, Hpost, Hres, u_save,
                 r_save);
    else
        launch_k(k_compute_h_fwd<N>, dim3(unsigned((T * N + 127) / 128)), dim3(128), 0, s, upart,
                 spart, S, alpha, b, T, K, iters, eps_sk, eps_rms, Hpre, Hpost, Hres, u_save,
                 r_save);
}

// The compute_h backward launch: partial rows of 128 / n tokens per block
template <int N>
static cudaError_t launch_ch_bwd(const float *dHpre, const float *dHpost, const float *dHres,
                                 const float *u_save, const float *r_save, const float *alpha,
                                 const float *b, int64_t T, int64_t K, int iters, float eps_sk,
                                 float eps_rms, bf16 *du_hl, int du_cols, float *coef,
                                 float *part, const float *s_tot, float *du_f32, float *dub,
                                 const float *Hres, float *HresT, cudaStream_t s)
{
    const int64_t prows = (T * N + 127) / 128;
    cudaError_t e;
    if constexpr (N == 4) {
        e = set_smem_limit(reinterpret_cast<const void *>(k_compute_h_bwd4),
                           int(size_t(8) * kMaxIters * kCh4Bwd * sizeof(float)));
        if (e != cudaSuccess) return e;
        if (du_cols != kCh4DuCols) return cudaErrorInvalidValue;
        MHC_PROF("k_compute_h_bwd", s);
        launch_k(k_compute_h_bwd4, dim3(unsigned(prows)), dim3(kCh4Bwd),
                 size_t(8) * iters * kCh4Bwd * sizeof(float), s, dHpre, dHpost, dHres, u_save,
                 r_save, alpha, b, T, K, iters, eps_sk, eps_rms, du_hl, coef, part, s_tot, du_f32,
                 dub);
    } else {
        e = set_smem_limit(reinterpret_cast<const void *>(k_compute_h_bwd<N>),
                           int(size_t(2) * kMaxIters * 128 * sizeof(float)));
        if (e != cudaSuccess) return e;
        MHC_PROF("k_compute_h_bwd", s);
        launch_k(k_compute_h_bwd<N>, dim3(unsigned(prows)), dim3(128),
                 size_t(2) * iters * 128 * sizeof(float), s, dHpre, dHpost, dHres, u_save, r_save,
                 alpha, b, T, K, iters, eps_sk, eps_rms, du_hl, du_cols, coef, part, s_tot, du_f32,
                 dub, Hres, HresT);
    }
    return cudaGetLastError();
}

// Fixed-order sums of the backward's partials.  Blocks [0, wblocks):
// dW[j] = sum_s dWpart[s][j]; the next bblocks: dbias[j] = sum_s
// dbiaspart[s][j] (s ascending; both only when the residual-gradient pass
// was split); then one block per column o of the partial rows: db[o] (o < O)
// or dalpha[o - O] = sum over rows, a fixed 256-thread tree.
__global__ void __launch_bounds__(256)
    k_bwd_finalize(const float *__restrict__ dWpart, float *__restrict__ dW, int64_t wcols,
                   int wblocks, const float *__restrict__ dbiaspart, float *__restrict__ dbias,
                   int64_t bcols, int bblocks, int splits, const float *__restrict__ part,
                   int64_t prows, int O, float *__restrict__ db, float *__restrict__ dalpha)
{
    pdl_wait();
    __shared__ float red[256];
    int blk = blockIdx.x;
    if (blk < wblocks + bblocks) {
        const bool isw = blk < wblocks;
        const float *src = isw ? dWpart : dbiaspart;
        float *dst = isw ? dW : dbias;
        const int64_t cols = isw ? wcols : bcols;
        const int64_t c = int64_t(isw ? blk : blk - wblocks) * 256 + threadIdx.x;
        if (c >= cols) return;
        float acc = 0.f;
        for (int sp = 0; sp < splits; ++sp) acc += src[int64_t(sp) * cols + c];
        dst[c] = acc;
        return;
    }
    const int o = blk - wblocks - bblocks;
    const int PW = O + 4;
    float acc = 0.f;
    for (int64_t r = threadIdx.x; r < prows; r += 256) acc += part[r * PW + o];
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        if (o < O)
            db[o] = red[0];
        else
            dalpha[o - O] = red[0];
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// forward workspace: W_hl [w_split_rows(n)][K] bf16, partials upart [S][T][O], spart [S][T]
size_t proj_fwd_ws_bytes(int64_t T, int n, int64_t C)
{
    const int64_t O = int64_t(n) * n + 2 * n, K = int64_t(n) * C;
    const int64_t S = proj_tc_splits(T, n, K);
    return ws_align(size_t(w_split_rows(n) * K) * 2) + ws_align(size_t(S * T * O) * 4) +
           ws_align(size_t(S * T) * 4);
}

template <int N>
static cudaError_t proj_fwd_impl(const bf16 *x, const float *W, const float *alpha,
                                 const float *b, int64_t T, int64_t C, int iters, float eps_sk,
                                 float eps_rms, float *Hpre, float *Hpost, float *Hres,
                                 float *u_save, float *r_save, void *ws, int *fault,
                                 cudaStream_t s)
{
    constexpr int O = Dims<N>::O;
    const int64_t K = int64_t(N) * C;
    const int64_t S = proj_tc_splits(T, N, K);
    char *p = static_cast<char *>(ws);
    bf16 *Whl = reinterpret_cast<bf16 *>(p);
    p += ws_align(size_t(w_split_rows(N) * K) * 2);
    float *upart = reinterpret_cast<float *>(p);
    p += ws_align(size_t(S * T * O) * 4);
    float *spart = reinterpret_cast<float *>(p);
    int S_used = 1;
    cudaError_t e = launch_proj_partials(x, W, T, N, C, Whl, upart, spart, &S_used, fault, s);
    if (e != cudaSuccess) return e;
    launch_ch_fwd<N>(upart, spart, S_used, alpha, b, T, K, iters, eps_sk, eps_rms, Hpre, Hpost, Hres,
                     u_save, r_save, s);
    return cudaGetLastError();
}

cudaError_t launch_compute_h_parts(const float *upart, const float *spart, int S,
                                   const float *alpha, const float *b, int64_t T, int n,
                                   int64_t C, int iters, float eps_sk, float eps_rms, float *Hpre,
                                   float *Hpost, float *Hres, float *u_save, float *r_save,
                                   cudaStream_t s)
{
    const int64_t K = int64_t(n) * C;
    if (n == 4)
        launch_ch_fwd<4>(upart, spart, S, alpha, b, T, K, iters, eps_sk, eps_rms, Hpre, Hpost,
                         Hres, u_save, r_save, s);
    else
        launch_ch_fwd<8>(upart, spart, S, alpha, b, T, K, iters, eps_sk, eps_rms, Hpre, Hpost,
                         Hres, u_save, r_save, s);
    return cudaGetLastError();
}

cudaError_t launch_proj_fwd(const bf16 *x, const float *W, const float *alpha, const float *b,
                            int64_t T, int n, int64_t C, int iters, float eps_sk, float eps_rms,
                            float *Hpre, float *Hpost, float *Hres, float *u_save, float *r_save,
                            void *ws, int *fault, cudaStream_t s)
{
    if (n == 4)
        return proj_fwd_impl<4>(x, W, alpha, b, T, C, iters, eps_sk, eps_rms, Hpre, Hpost, Hres,
                                u_save, r_save, ws, fault, s);
    return proj_fwd_impl<8>(x, W, alpha, b, T, C, iters, eps_sk, eps_rms, Hpre, Hpost, Hres,
                            u_save, r_save, ws, fault, s);
}

// workspace layout of the backward (each piece 256-byte aligned):
//   du_hl [T][du_cols] bf16, du [T][O] fp32, dub [T], coef [T], partial rows
//   [ceil(T n / 128)][n*n+2n+4], dH_pre, dH_post [T][n], dH_res [T][n][n]
//   (layer), dbias partials [S][C], dW partials [S][K][O] (only when S > 1)
struct BwdWs {
    bf16 *du_hl;
    float *du32, *dub, *coef, *part, *dHpre, *dHpost, *dHres, *HresT, *dWpart, *dbiaspart;
    int splits;
    size_t bytes;
};

static BwdWs carve_bwd(void *base, int64_t T, int n, int64_t C)
{
    const int64_t O = int64_t(n) * n + 2 * n, K = int64_t(n) * C;
    BwdWs w;
    char *p = static_cast<char *>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        char *q = p ? p + off : nullptr;
        off += ws_align(bytes);
        return q;
    };
    w.splits = bwd_tc_splits(T, n, C);
    w.du_hl = reinterpret_cast<bf16 *>(take(size_t(T) * bwd_tc_du_cols(n) * 2));
    w.du32 = reinterpret_cast<float *>(take(size_t(T * O) * 4));
    w.dub = reinterpret_cast<float *>(take(size_t(T) * 4));
    w.coef = reinterpret_cast<float *>(take(size_t(T) * 4));
    w.part = reinterpret_cast<float *>(take(size_t((T * n + 127) / 128) * bwd_part_cols(n) * 4));
    w.dHpre = reinterpret_cast<float *>(take(size_t(T * n) * 4));
    w.dHpost = reinterpret_cast<float *>(take(size_t(T * n) * 4));
    w.dHres = reinterpret_cast<float *>(take(size_t(T * n * n) * 4));
    w.HresT = n == 8 ? reinterpret_cast<float *>(take(size_t(T * n * n) * 4)) : nullptr;
    w.dbiaspart = reinterpret_cast<float *>(take(size_t(w.splits) * size_t(C) * 4));
    w.dWpart = w.splits > 1 ? reinterpret_cast<float *>(take(size_t(w.splits) * size_t(K * O) * 4))
                            : nullptr;
    w.bytes = off;
    return w;
}

size_t proj_bwd_ws_bytes(int64_t T, int n, int64_t C) { return carve_bwd(nullptr, T, n, C).bytes; }

struct LayerBwd {
    const bf16 *dout, *dy, *f, *bias;
    const float *Hpre, *Hpost, *Hres;
    bf16 *df;
    float *dbias;
};

template <int N>
static cudaError_t bwd_impl(const float *dHpre, const float *dHpost, const float *dHres,
                            const bf16 *x, const float *W, const float *alpha, const float *b,
                            const float *u_save, const float *r_save, int64_t T, int64_t C,
                            int iters, float eps_sk, float eps_rms, const LayerBwd *L, bf16 *dx,
                            float *dW, float *dalpha, float *db, void *ws, int *fault,
                            cudaStream_t s)
{
    constexpr int O = Dims<N>::O;
    const int64_t K = int64_t(N) * C;
    const int du_cols = bwd_tc_du_cols(N);
    BwdWs w = carve_bwd(ws, T, N, C);
    cudaError_t e;
    if (L) {
        // pass 1: per-token sums over dout, x, f, dy and df
        e = launch_bwd_tok(L->dout, x, L->f, L->bias, L->dy, L->Hpost, T, N, C, L->df, w.dHres,
                           w.dHpost, w.dHpre, s);
        if (e != cudaSuccess) return e;
        dHpre = w.dHpre;
        dHpost = w.dHpost;
        dHres = w.dHres;
    }
    const int64_t prows = (T * N + 127) / 128;
    // n = 8 (layer): H_res transposed for the residual-gradient pass's mix
    const bool hT = L && N == 8;
    e = launch_ch_bwd<N>(dHpre, dHpost, dHres, u_save, r_save, alpha, b, T, K, iters, eps_sk,
                         eps_rms, w.du_hl, du_cols, w.coef, w.part, nullptr, w.du32, w.dub,
                         hT ? L->Hres : nullptr, hT ? w.HresT : nullptr, s);
    if (e != cudaSuccess) return e;
    // pass 2: residual gradient, dW and dbias on the tensor cores; an unsplit
    // pass writes dW and dbias directly
    const int tiles = int((T + 127) / 128);
    const int tps = (tiles + w.splits - 1) / w.splits;
    const int splits_used = (tiles + tps - 1) / tps;
    const bool split = splits_used > 1;
    float *dbias = L ? L->dbias : nullptr;
    e = launch_bwd_tc(x, W, w.du_hl, w.du32, w.dub, w.coef, T, N, C, L ? L->dout : nullptr,
                      L ? L->dy : nullptr,
                      L ? L->Hpre : nullptr, L ? (hT ? w.HresT : L->Hres) : nullptr,
                      L ? L->Hpost : nullptr, dx,
                      split ? w.dWpart : dW, (split || !dbias) ? w.dbiaspart : dbias,
                      splits_used, fault, s);
    if (e != cudaSuccess) return e;
    const int wblocks = split ? int((K * O + 255) / 256) : 0;
    const int bblocks = (split && dbias) ? int((C + 255) / 256) : 0;
    {
        MHC_PROF("k_bwd_finalize", s);
        launch_k(k_bwd_finalize, dim3(unsigned(wblocks + bblocks + O + 3)), dim3(256), 0, s, 
            w.dWpart, dW, K * O, wblocks, w.dbiaspart, dbias, C, bblocks, splits_used, w.part,
            prows, O, db, dalpha);
    }
    return cudaGetLastError();
}

cudaError_t launch_proj_bwd(const float *dHpre, const float *dHpost, const float *dHres,
                            const bf16 *x, const float *W, const float *alpha, const float *b,
                            const float *u_save, const float *r_save, int64_t T, int n,
                            int64_t C, int iters, float eps_sk, float eps_rms, bf16 *dx,
                            float *dW, float *dalpha, float *db, void *ws, int *fault,
                            cudaStream_t s)
{
    if (n == 4)
        return bwd_impl<4>(dHpre, dHpost, dHres, x, W, alpha, b, u_save, r_save, T, C, iters,
                           eps_sk, eps_rms, nullptr, dx, dW, dalpha, db, ws, fault, s);
    return bwd_impl<8>(dHpre, dHpost, dHres, x, W, alpha, b, u_save, r_save, T, C, iters,
                       eps_sk, eps_rms, nullptr, dx, dW, dalpha, db, ws, fault, s);
}

cudaError_t launch_layer_bwd(const bf16 *dout, const bf16 *dy, const bf16 *x, const float *W,
                             const float *alpha, const float *b, const bf16 *f,
                             const bf16 *bias, const float *Hpre, const float *Hpost,
                             const float *Hres, const float *u_save, const float *r_save,
                             int64_t T, int n, int64_t C, int iters, float eps_sk,
                             float eps_rms, bf16 *dx, bf16 *df, float *dW, float *dalpha,
                             float *db, float *dbias, void *ws, int *fault, cudaStream_t s)
{
    const LayerBwd L{dout, dy, f, bias, Hpre, Hpost, Hres, df, dbias};
    if (n == 4)
        return bwd_impl<4>(nullptr, nullptr, nullptr, x, W, alpha, b, u_save, r_save, T, C,
                           iters, eps_sk, eps_rms, &L, dx, dW, dalpha, db, ws, fault, s);
    return bwd_impl<8>(nullptr, nullptr, nullptr, x, W, alpha, b, u_save, r_save, T, C, iters,
                       eps_sk, eps_rms, &L, dx, dW, dalpha, db, ws, fault, s);
}

// ---------------------------------------------------------------------------
// proj_rms_compute_h over channel shards (RL-Kernel PR #383 task P1-6, the
// fp32_gemm_rms TP/SP contract): a shard's partial sums, compute_h on the
// totals, the per-token backward coefficients, a shard's dx and dW.
// ---------------------------------------------------------------------------
// u[t][o] = sum_s upart[s][t][o], s[t] = sum_s spart[s][t] (s ascending)
__global__ void k_sum_splits(const float *__restrict__ upart, const float *__restrict__ spart,
                             int S, int64_t T, int O, float *__restrict__ u,
                             float *__restrict__ s_out)
{
    pdl_wait();
    const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t TO = T * O;
    if (e < TO) {
        float a = 0.f;
        for (int sp = 0; sp < S; ++sp) a += upart[int64_t(sp) * TO + e];
        u[e] = a;
    } else if (e < TO + T) {
        const int64_t t = e - TO;
        float a = 0.f;
        for (int sp = 0; sp < S; ++sp) a += spart[int64_t(sp) * T + t];
        s_out[t] = a;
    }
}

cudaError_t launch_proj_partial_sums(const bf16 *x, const float *W, int64_t T, int n, int64_t Cs,
                                     float *u, float *s_out, void *ws, int *fault, cudaStream_t s)
{
    const int64_t O = int64_t(n) * n + 2 * n, K = int64_t(n) * Cs;
    const int64_t S = proj_tc_splits(T, n, K);
    char *p = static_cast<char *>(ws);
    bf16 *Whl = reinterpret_cast<bf16 *>(p);
    p += ws_align(size_t(w_split_rows(n) * K) * 2);
    float *upart = reinterpret_cast<float *>(p);
    p += ws_align(size_t(S * T * O) * 4);
    float *spart = reinterpret_cast<float *>(p);
    int S_used = 1;
    cudaError_t e = launch_proj_partials(x, W, T, n, Cs, Whl, upart, spart, &S_used, fault, s);
    if (e != cudaSuccess) return e;
    MHC_PROF("k_sum_splits", s);
    launch_k(k_sum_splits, dim3(unsigned((T * O + T + 255) / 256)), dim3(256), 0, s, upart, spart, S_used, T,
                                                                   int(O), u, s_out);
    return cudaGetLastError();
}

cudaError_t launch_compute_h_fwd(const float *u, const float *s_tot, int64_t K,
                                 const float *alpha, const float *b, int64_t T, int n, int iters,
                                 float eps_sk, float eps_rms, float *Hpre, float *Hpost,
                                 float *Hres, float *r_save, cudaStream_t s)
{
    if (n == 4)
        launch_ch_fwd<4>(u, s_tot, 1, alpha, b, T, K, iters, eps_sk, eps_rms, Hpre, Hpost, Hres,
                         nullptr, r_save, s);
    else
        launch_ch_fwd<8>(u, s_tot, 1, alpha, b, T, K, iters, eps_sk, eps_rms, Hpre, Hpost, Hres,
                         nullptr, r_save, s);
    return cudaGetLastError();
}

// scratch of the sharded compute_h backward: du_hl [T][du_cols], partial rows
size_t compute_h_bwd_ws_bytes(int64_t T, int n)
{
    return ws_align(size_t(T) * bwd_tc_du_cols(n) * 2) +
           ws_align(size_t((T * n + 127) / 128) * bwd_part_cols(n) * 4);
}

template <int N>
static cudaError_t compute_h_bwd_impl(const float *dHpre, const float *dHpost,
                                      const float *dHres, const float *u, const float *s_tot,
                                      int64_t K, const float *alpha, const float *b, int64_t T,
                                      int iters, float eps_sk, float eps_rms, float *du,
                                      float *coef, float *dalpha, float *db, void *ws,
                                      cudaStream_t s)
{
    constexpr int O = Dims<N>::O;
    char *p = static_cast<char *>(ws);
    bf16 *du_hl = reinterpret_cast<bf16 *>(p);
    p += ws_align(size_t(T) * bwd_tc_du_cols(N) * 2);
    float *part = reinterpret_cast<float *>(p);
    const int64_t prows = (T * N + 127) / 128;
    cudaError_t e = launch_ch_bwd<N>(dHpre, dHpost, dHres, u, nullptr, alpha, b, T, K, iters,
                                     eps_sk, eps_rms, du_hl, bwd_tc_du_cols(N), coef, part, s_tot,
                                     du, nullptr, nullptr, nullptr, s);
    if (e != cudaSuccess) return e;
    {
        MHC_PROF("k_bwd_finalize", s);
        launch_k(k_bwd_finalize, dim3(unsigned(O + 3)), dim3(256), 0, s, nullptr, nullptr, 0, 0, nullptr, nullptr, 0,
                                                        0, 1, part, prows, O, db, dalpha);
    }
    return cudaGetLastError();
}

cudaError_t launch_compute_h_bwd(const float *dHpre, const float *dHpost, const float *dHres,
                                 const float *u, const float *s_tot, int64_t K,
                                 const float *alpha, const float *b, int64_t T, int n, int iters,
                                 float eps_sk, float eps_rms, float *du, float *coef,
                                 float *dalpha, float *db, void *ws, cudaStream_t s)
{
    if (n == 4)
        return compute_h_bwd_impl<4>(dHpre, dHpost, dHres, u, s_tot, K, alpha, b, T, iters,
                                     eps_sk, eps_rms, du, coef, dalpha, db, ws, s);
    return compute_h_bwd_impl<8>(dHpre, dHpost, dHres, u, s_tot, K, alpha, b, T, iters, eps_sk,
                                 eps_rms, du, coef, dalpha, db, ws, s);
}

// du (fp32 [T][O]) -> du_hl rows: bf16 hi | lo, zeros for the rest of the
// row; the element at column 0 also writes dub[t] = sum_o |du[t][o]|
__global__ void k_du_split(const float *__restrict__ du, int64_t T, int O, int du_cols,
                           bf16 *__restrict__ du_hl, float *__restrict__ dub)
{
    pdl_wait();
    const int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (e >= T * du_cols) return;
    const int64_t t = e / du_cols;
    const int c = int(e % du_cols);
    if (c == 0) {
        float sabs = 0.f;
        for (int o = 0; o < O; ++o) sabs += fabsf(__ldg(du + t * O + o));
        dub[t] = sabs;
    }
    bf16 v = __float2bfloat16_rn(0.f);
    if (c < 2 * O) {
        const float d = __ldg(du + t * O + (c % O));
        const bf16 hi = __float2bfloat16_rn(d);
        v = c < O ? hi : __float2bfloat16_rn(d - __bfloat162float(hi));
    }
    du_hl[e] = v;
}

size_t proj_partial_bwd_ws_bytes(int64_t T, int n, int64_t Cs) { return proj_bwd_ws_bytes(T, n, Cs); }

cudaError_t launch_proj_partial_bwd(const bf16 *x, const float *W, const float *du,
                                    const float *coef, int64_t T, int n, int64_t Cs, bf16 *dx,
                                    float *dW, void *ws, int *fault, cudaStream_t s)
{
    const int64_t O = int64_t(n) * n + 2 * n, K = int64_t(n) * Cs;
    BwdWs w = carve_bwd(ws, T, n, Cs);
    const int du_cols = bwd_tc_du_cols(n);
    {
        MHC_PROF("k_du_split", s);
        launch_k(k_du_split, dim3(unsigned((T * du_cols + 255) / 256)), dim3(256), 0, s, du, T,
                 int(O), du_cols, w.du_hl, w.dub);
    }
    const int tiles = int((T + 127) / 128);
    const int tps = (tiles + w.splits - 1) / w.splits;
    const int splits_used = (tiles + tps - 1) / tps;
    const bool split = splits_used > 1;
    cudaError_t e = launch_bwd_tc(x, W, w.du_hl, du, w.dub, coef, T, n, Cs, nullptr, nullptr, nullptr,
                                  nullptr, nullptr, dx, split ? w.dWpart : dW, w.dbiaspart,
                                  splits_used, fault, s);
    if (e != cudaSuccess) return e;
    if (split) {
        const int wblocks = int((K * O + 255) / 256);
        MHC_PROF("k_bwd_finalize", s);
        launch_k(k_bwd_finalize, dim3(unsigned(wblocks)), dim3(256), 0, s, w.dWpart, dW, K * O, wblocks, nullptr,
                                                          nullptr, 0, 0, splits_used, nullptr, 0,
                                                          int(O), nullptr, nullptr);
    }
    return cudaGetLastError();
}

}  // namespace mhc
