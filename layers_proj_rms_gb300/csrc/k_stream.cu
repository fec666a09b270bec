// HBM-streaming kernels of the mHC layer: h_aggregate fwd/bwd, h_post_bda
// fwd/bwd (per-token part and the dbias column sum) and the standalone
// RMSNorm fwd/bwd.  Every global access is a 16-byte vector of 8 bf16
// values; all sums are fp32 in a fixed order (no atomics).
//
// Definitions: Megatron-Core fused_mhc_kernels (fused_h_aggregate,
// _torch_h_aggregate_bwd, fused_h_post_bda "H_res.T @ residual + H_post *
// (x + bias)", _torch_h_post_bda_bwd) and rwkv-ops mhu_ffi.cu
// (StreamAggregateFwd/Bwd, MhcPostOpFwdHost/BwdHost, RMSNormFwdHost/BwdHost).
#include <atomic>
#include <mutex>
#include <vector>

#include "launch.h"

namespace mhc {

// SM count per device, looked up once; relaxed atomics so that threads
// calling concurrently race on nothing (two first calls may both look it up
// and store the same value).
static std::atomic<int> g_num_sms[64];

int num_sms()
{
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    int v = g_num_sms[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        if (v <= 0) v = 1;
        g_num_sms[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

cudaError_t set_smem_limit(const void *kernel, int bytes)
{
    struct Entry {
        int dev;
        const void *kernel;
        int bytes;
    };
    static std::mutex mu;
    static std::vector<Entry> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    for (const Entry &d : done)
        if (d.dev == dev && d.kernel == kernel && d.bytes >= bytes) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.push_back({dev, kernel, bytes});
    return e;
}

static unsigned grid_for(int64_t work, int per_sm)
{
    const int64_t cap = int64_t(num_sms()) * per_sm;
    return unsigned(work < cap ? (work > 0 ? work : 1) : cap);
}

static int threads_for(int64_t C8)
{
    int t = int((C8 + 31) / 32) * 32;
    return t < 256 ? t : 256;
}

// ---------------------------------------------------------------------------
// h_aggregate forward: y[t][c] = sum_i H_pre[t][i] x[t][i][c]
// One block walks tokens; each thread one 8-wide chunk of c at a time.
// ---------------------------------------------------------------------------
template <int N, bool STATIC>
__global__ void __launch_bounds__(256)
    k_agg_fwd(const bf16 *__restrict__ x, const float *__restrict__ Hpre, bf16 *__restrict__ y,
              int64_t T, int64_t C8)
{
    pdl_wait();
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        float h[N];
#pragma unroll
        for (int i = 0; i < N; ++i) h[i] = __ldg(Hpre + (STATIC ? 0 : t * N) + i);
        for (int64_t c8 = threadIdx.x; c8 < C8; c8 += blockDim.x) {
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < N; ++i) {
                float v[8];
                unpack8(ld_stream(x + ((t * N + i) * C8 + c8) * 8), v);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = fmaf(h[i], v[e], acc[e]);
            }
            st_stream(y + (t * C8 + c8) * 8, pack8(acc));
        }
    }
}

// ---------------------------------------------------------------------------
// h_aggregate backward: dx[t][i][c] = H_pre[t][i] dy[t][c] (if dx != null),
// dH_pre[t][i] = sum_c dy[t][c] x[t][i][c].  One warp per token; each lane
// keeps U chunks of 8 channels (with all n streams) in flight.
// ---------------------------------------------------------------------------
template <int N>
__global__ void __launch_bounds__(256)
    k_agg_bwd(const bf16 *__restrict__ dy, const bf16 *__restrict__ x,
              const float *__restrict__ Hpre, bf16 *__restrict__ dx, float *__restrict__ dHpre,
              int64_t T, int64_t C8)
{
    pdl_wait();
    constexpr int U = N == 4 ? 4 : 2;
    const int lane = threadIdx.x & 31;
    const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
    for (int64_t t = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T;
         t += warps) {
        float h[N], part[N];
#pragma unroll
        for (int i = 0; i < N; ++i) {
            h[i] = __ldg(Hpre + t * N + i);
            part[i] = 0.f;
        }
        for (int64_t base = lane; base < C8; base += 32 * U) {
            uint4 gv[U], xv[U][N];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c8 = base + 32 * u;
                if (c8 < C8) {
                    gv[u] = ld_stream(dy + (t * C8 + c8) * 8);
#pragma unroll
                    for (int i = 0; i < N; ++i) xv[u][i] = ld_stream(x + ((t * N + i) * C8 + c8) * 8);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c8 = base + 32 * u;
                if (c8 >= C8) continue;
                float g[8];
                unpack8(gv[u], g);
#pragma unroll
                for (int i = 0; i < N; ++i) {
                    float v[8];
                    unpack8(xv[u][i], v);
                    float acc = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc = fmaf(g[e], v[e], acc);
                    part[i] += acc;
                    if (dx) {
                        float o[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = h[i] * g[e];
                        st_stream(dx + ((t * N + i) * C8 + c8) * 8, pack8(o));
                    }
                }
            }
        }
#pragma unroll
        for (int i = 0; i < N; ++i) part[i] = warp_sum(part[i]);
        if (lane == 0)
#pragma unroll
            for (int i = 0; i < N; ++i) dHpre[t * N + i] = part[i];
    }
}

// ---------------------------------------------------------------------------
// h_aggregate backward with one static H_pre [N] (rwkv-ops StreamAggregateBwd
// with per_token = false): dx[t][i][c] = H_pre[i] dy[t][c] (if dx != null),
// dH_pre[i] = sum_t sum_c dy x_i.  Warp per token as in k_agg_bwd; each warp
// keeps its running sums over its tokens (ascending), the block adds its
// warps in order and writes one partial row part[block][N]; k_col_sum adds
// the rows in block order.
// ---------------------------------------------------------------------------
template <int N>
__global__ void __launch_bounds__(256)
    k_agg_bwd_static(const bf16 *__restrict__ dy, const bf16 *__restrict__ x,
                     const float *__restrict__ Hpre, bf16 *__restrict__ dx,
                     float *__restrict__ part, int64_t T, int64_t C8)
{
    pdl_wait();
    __shared__ float red[8][N];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
    float h[N], tot[N];
#pragma unroll
    for (int i = 0; i < N; ++i) {
        h[i] = __ldg(Hpre + i);
        tot[i] = 0.f;
    }
    for (int64_t t = int64_t(blockIdx.x) * (blockDim.x >> 5) + warp; t < T; t += warps) {
        float p[N];
#pragma unroll
        for (int i = 0; i < N; ++i) p[i] = 0.f;
        for (int64_t c8 = lane; c8 < C8; c8 += 32) {
            float g[8];
            unpack8(ld_stream(dy + (t * C8 + c8) * 8), g);
#pragma unroll
            for (int i = 0; i < N; ++i) {
                float v[8];
                unpack8(ld_stream(x + ((t * N + i) * C8 + c8) * 8), v);
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc = fmaf(g[e], v[e], acc);
                p[i] += acc;
                if (dx) {
                    float o[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) o[e] = h[i] * g[e];
                    st_stream(dx + ((t * N + i) * C8 + c8) * 8, pack8(o));
                }
            }
        }
#pragma unroll
        for (int i = 0; i < N; ++i) tot[i] += warp_sum(p[i]);
    }
    if (lane == 0)
#pragma unroll
        for (int i = 0; i < N; ++i) red[warp][i] = tot[i];
    __syncthreads();
    if (threadIdx.x < N) {
        float s = 0.f;
        for (int w = 0; w < int(blockDim.x >> 5); ++w) s += red[w][threadIdx.x];
        part[int64_t(blockIdx.x) * N + threadIdx.x] = s;
    }
}

// ---------------------------------------------------------------------------
// h_post_bda forward:
//   out[t][i][c] = sum_j H_res[t][j][i] res[t][j][c] + H_post[t][i] (f[t][c] + bias[c])
// One warp per token; each lane keeps U chunks of 8 channels in flight.
// ---------------------------------------------------------------------------
template <int N>
__global__ void __launch_bounds__(256)
    k_post_fwd(const bf16 *__restrict__ res, const bf16 *__restrict__ f,
               const bf16 *__restrict__ bias, const float *__restrict__ Hres,
               const float *__restrict__ Hpost, bf16 *__restrict__ out, int64_t T, int64_t C8)
{
    pdl_wait();
    constexpr int U = N == 4 ? 2 : 1;
    const int lane = threadIdx.x & 31;
    const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
    for (int64_t t = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T;
         t += warps) {
        float hr[N * N], hp[N];
#pragma unroll
        for (int e = 0; e < N * N; e += 4) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(Hres + t * N * N + e));
            hr[e] = v.x;
            hr[e + 1] = v.y;
            hr[e + 2] = v.z;
            hr[e + 3] = v.w;
        }
#pragma unroll
        for (int i = 0; i < N; ++i) hp[i] = __ldg(Hpost + t * N + i);
        for (int64_t base = lane; base < C8; base += 32 * U) {
            uint4 fv[U], bv[U], xr[U][N];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c8 = base + 32 * u;
                if (c8 < C8) {
                    fv[u] = ld_stream(f + (t * C8 + c8) * 8);
                    bv[u] = bias ? __ldg(reinterpret_cast<const uint4 *>(bias + c8 * 8))
                                 : make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int j = 0; j < N; ++j) xr[u][j] = ld_stream(res + ((t * N + j) * C8 + c8) * 8);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c8 = base + 32 * u;
                if (c8 >= C8) continue;
                float fb[8], bb[8];
                unpack8(fv[u], fb);
                unpack8(bv[u], bb);
#pragma unroll
                for (int e = 0; e < 8; ++e) fb[e] += bb[e];
                float acc[N][8];
#pragma unroll
                for (int i = 0; i < N; ++i)
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[i][e] = hp[i] * fb[e];
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    float v[8];
                    unpack8(xr[u][j], v);
#pragma unroll
                    for (int i = 0; i < N; ++i)
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(hr[j * N + i], v[e], acc[i][e]);
                }
#pragma unroll
                for (int i = 0; i < N; ++i) st_stream(out + ((t * N + i) * C8 + c8) * 8, pack8(acc[i]));
            }
        }
    }
}

// n = 8: the eight 8-channel accumulators and the 8x8 H_res in registers
// (170 per thread) left one 256-thread block per SM and ~37 KB of loads in
// flight.  Here the warp's H_res and H_post rows sit in shared memory (read
// at uniform addresses), the outputs are formed in two halves of four (the
// same operations in the same order per output), each lane keeps U chunks in
// flight, and blocks are 4 warps.
template <int U>
__global__ void __launch_bounds__(128, 4)
    k_post_fwd8(const bf16 *__restrict__ res, const bf16 *__restrict__ f,
                const bf16 *__restrict__ bias, const float *__restrict__ Hres,
                const float *__restrict__ Hpost, bf16 *__restrict__ out, int64_t T, int64_t C8)
{
    constexpr int N = 8;
    pdl_wait();
    __shared__ float4 hsm[4][18];   // per warp: H_res[t] (16 float4), H_post[t] (2 float4)
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
    for (int64_t t = int64_t(blockIdx.x) * (blockDim.x >> 5) + w; t < T; t += warps) {
        __syncwarp();
        if (lane < 16)
            hsm[w][lane] = __ldg(reinterpret_cast<const float4 *>(Hres + t * N * N) + lane);
        else if (lane < 18)
            hsm[w][lane] = __ldg(reinterpret_cast<const float4 *>(Hpost + t * N) + (lane - 16));
        __syncwarp();
        for (int64_t base = lane; base < C8; base += 32 * U) {
            uint4 fv[U], bv[U], xr[U][N];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c8 = base + 32 * u;
                if (c8 < C8) {
                    fv[u] = ld_stream(f + (t * C8 + c8) * 8);
                    bv[u] = bias ? __ldg(reinterpret_cast<const uint4 *>(bias + c8 * 8))
                                 : make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int j = 0; j < N; ++j) xr[u][j] = ld_stream(res + ((t * N + j) * C8 + c8) * 8);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c8 = base + 32 * u;
                if (c8 >= C8) continue;
                float fb[8], bb[8];
                unpack8(fv[u], fb);
                unpack8(bv[u], bb);
#pragma unroll
                for (int e = 0; e < 8; ++e) fb[e] += bb[e];
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const float4 hp4 = hsm[w][16 + half];
                    const float hp[4] = {hp4.x, hp4.y, hp4.z, hp4.w};
                    float acc[4][8];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[i][e] = hp[i] * fb[e];
#pragma unroll
                    for (int j = 0; j < N; ++j) {
                        float v[8];
                        unpack8(xr[u][j], v);
                        const float4 h4 = hsm[w][2 * j + half];   // H_res[t][j][4 half .. 4 half + 3]
                        const float hr[4] = {h4.x, h4.y, h4.z, h4.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i)
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(hr[i], v[e], acc[i][e]);
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        st_stream(out + ((t * N + 4 * half + i) * C8 + c8) * 8, pack8(acc[i]));
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// h_post_bda backward, per-token part.  One warp per token:
//   dres[t][j][c]  = sum_i H_res[t][j][i] dout[t][i][c]     (if dres != null)
//   df[t][c]       = sum_i H_post[t][i] dout[t][i][c]        (if df != null)
//   dH_res[t][j][i] = sum_c res[t][j][c] dout[t][i][c]
//   dH_post[t][i]  = sum_c dout[t][i][c] (f[t][c] + bias[c])
// ---------------------------------------------------------------------------
template <int N>
__global__ void __launch_bounds__(256)
    k_post_bwd_tok(const bf16 *__restrict__ dout, const bf16 *__restrict__ res,
                   const bf16 *__restrict__ f, const bf16 *__restrict__ bias,
                   const float *__restrict__ Hres, const float *__restrict__ Hpost,
                   bf16 *__restrict__ dres, bf16 *__restrict__ df, float *__restrict__ dHres,
                   float *__restrict__ dHpost, int64_t T, int64_t C8)
{
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
    for (int64_t t = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T;
         t += warps) {
        const float *hr = Hres + t * N * N;  // read through L1 where used
        float hp[N];
#pragma unroll
        for (int i = 0; i < N; ++i) hp[i] = __ldg(Hpost + t * N + i);
        float aR[N * N], aP[N];
#pragma unroll
        for (int e = 0; e < N * N; ++e) aR[e] = 0.f;
#pragma unroll
        for (int i = 0; i < N; ++i) aP[i] = 0.f;
        for (int64_t c8 = lane; c8 < C8; c8 += 32) {
            uint4 dr[N], xr[N];
#pragma unroll
            for (int i = 0; i < N; ++i) dr[i] = ld_stream(dout + ((t * N + i) * C8 + c8) * 8);
#pragma unroll
            for (int j = 0; j < N; ++j) xr[j] = ld_stream(res + ((t * N + j) * C8 + c8) * 8);
            float fb[8];
            unpack8(ld_stream(f + (t * C8 + c8) * 8), fb);
            if (bias) {
                float bv[8];
                unpack8(__ldg(reinterpret_cast<const uint4 *>(bias + c8 * 8)), bv);
#pragma unroll
                for (int e = 0; e < 8; ++e) fb[e] += bv[e];
            }
            float dfv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < N; ++i) {
                float d[8];
                unpack8(dr[i], d);
                float sp = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    sp = fmaf(d[e], fb[e], sp);
                    dfv[e] = fmaf(hp[i], d[e], dfv[e]);
                }
                aP[i] += sp;
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    float v[8];
                    unpack8(xr[j], v);
                    float s = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) s = fmaf(v[e], d[e], s);
                    aR[j * N + i] += s;
                }
            }
            if (df) st_stream(df + (t * C8 + c8) * 8, pack8(dfv));
            if (dres) {
#pragma unroll
                for (int j = 0; j < N; ++j) {
                    float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int i = 0; i < N; ++i) {
                        float d[8];
                        unpack8(dr[i], d);
#pragma unroll
                        const float w = __ldg(hr + j * N + i);
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = fmaf(w, d[e], o[e]);
                    }
                    st_stream(dres + ((t * N + j) * C8 + c8) * 8, pack8(o));
                }
            }
        }
#pragma unroll
        for (int e = 0; e < N * N; ++e) aR[e] = warp_sum(aR[e]);
#pragma unroll
        for (int i = 0; i < N; ++i) aP[i] = warp_sum(aP[i]);
        if (lane == 0) {
#pragma unroll
            for (int e = 0; e < N * N; ++e) dHres[t * N * N + e] = aR[e];
#pragma unroll
            for (int i = 0; i < N; ++i) dHpost[t * N + i] = aP[i];
        }
    }
}

// ---------------------------------------------------------------------------
// dbias[c] = sum_t sum_i H_post[t][i] dout[t][i][c]: every thread owns one
// 8-wide chunk of c and a contiguous token range; partials per range are
// then summed in ascending range order.
// ---------------------------------------------------------------------------
static int64_t dbias_splits(int64_t T, int64_t C8)
{
    const int64_t cblocks = (C8 + 255) / 256;
    int64_t s = (int64_t(kSplitSms) * 4 + cblocks - 1) / cblocks;
    if (s > T) s = T;
    if (s > 256) s = 256;
    return s < 1 ? 1 : s;
}

size_t dbias_ws_bytes(int64_t T, int64_t C)
{
    return ws_align(size_t(dbias_splits(T, C / 8)) * size_t(C) * sizeof(float));
}

template <int N>
__global__ void __launch_bounds__(256)
    k_dbias_partial(const bf16 *__restrict__ dout, const float *__restrict__ Hpost,
                    float *__restrict__ part, int64_t T, int64_t C8, int64_t splits)
{
    pdl_wait();
    const int64_t c8 = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t s = blockIdx.y;
    const int64_t t0 = T * s / splits, t1 = T * (s + 1) / splits;
    if (c8 >= C8) return;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    for (int64_t t = t0; t < t1; ++t) {
        float dfv[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < N; ++i) {
            const float h = __ldg(Hpost + t * N + i);
            float d[8];
            unpack8(ld_stream(dout + ((t * N + i) * C8 + c8) * 8), d);
#pragma unroll
            for (int e = 0; e < 8; ++e) dfv[e] = fmaf(h, d[e], dfv[e]);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += dfv[e];
    }
    float4 *p = reinterpret_cast<float4 *>(part + (s * C8 + c8) * 8);
    p[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    p[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

__global__ void k_sum_rows(const float *__restrict__ part, float *__restrict__ out, int64_t rows,
                           int64_t cols)
{
    pdl_wait();
    const int64_t c = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (c >= cols) return;
    float acc = 0.f;
    for (int64_t r = 0; r < rows; ++r) acc += part[r * cols + c];
    out[c] = acc;
}

cudaError_t launch_dbias(const bf16 *dout, const float *Hpost, float *dbias, int64_t T, int n,
                         int64_t C, void *ws, cudaStream_t s)
{
    const int64_t C8 = C / 8;
    const int64_t splits = dbias_splits(T, C8);
    float *part = static_cast<float *>(ws);
    dim3 grid(unsigned((C8 + 255) / 256), unsigned(splits));
    if (n == 4) {
        MHC_PROF("k_dbias_partial", s);
        launch_k(k_dbias_partial<4>, dim3(grid), dim3(256), 0, s, dout, Hpost, part, T, C8, splits);
    } else {
        MHC_PROF("k_dbias_partial", s);
        launch_k(k_dbias_partial<8>, dim3(grid), dim3(256), 0, s, dout, Hpost, part, T, C8, splits);
    }
    {
        MHC_PROF("k_sum_rows", s);
        launch_k(k_sum_rows, dim3(unsigned((C + 255) / 256)), dim3(256), 0, s, part, dbias, splits, C);
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Standalone RMSNorm, one block per row, the row held in registers
// (R chunks of 8 values per thread).
//   fwd: rho = 1/sqrt(sum x^2 / cols + eps), y = x rho
//   bwd: dx = rho dy - rho^3 x (sum dy x) / cols
// ---------------------------------------------------------------------------
__device__ __forceinline__ float block_sum(float v, float *red)
{
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[w] = v;
    __syncthreads();
    float r = 0.f;
    const int nw = blockDim.x >> 5;
    for (int i = 0; i < nw; ++i) r += red[i];
    return r;
}

// Rows of at most 32*R chunks: one warp per row, the row in registers.
template <int R>
__global__ void __launch_bounds__(256)
    k_rms_fwd_w(const bf16 *__restrict__ x, bf16 *__restrict__ y, float *__restrict__ rstd,
                int64_t rows, int64_t C8, float inv_cols, float eps)
{
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
    for (int64_t r = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
         r += warps) {
        uint4 v[R];
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const int64_t c8 = lane + 32 * q;
            if (c8 < C8) v[q] = ld_stream(x + (r * C8 + c8) * 8);
        }
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const int64_t c8 = lane + 32 * q;
            if (c8 < C8) {
                float f[8];
                unpack8(v[q], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) s = fmaf(f[e], f[e], s);
            }
        }
        s = warp_sum(s);
        const float rho = rsqrtf(s * inv_cols + eps);
        if (rstd && lane == 0) rstd[r] = rho;
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const int64_t c8 = lane + 32 * q;
            if (c8 < C8) {
                float f[8];
                unpack8(v[q], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] *= rho;
                st_stream(y + (r * C8 + c8) * 8, pack8(f));
            }
        }
    }
}

template <int R>
__global__ void __launch_bounds__(256)
    k_rms_bwd_w(const bf16 *__restrict__ dy, const bf16 *__restrict__ x,
                const float *__restrict__ rstd, bf16 *__restrict__ dx, int64_t rows, int64_t C8,
                float inv_cols, float eps)
{
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t warps = int64_t(gridDim.x) * (blockDim.x >> 5);
    for (int64_t r = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows;
         r += warps) {
        uint4 vx[R], vg[R];
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const int64_t c8 = lane + 32 * q;
            if (c8 < C8) {
                vx[q] = ld_stream(x + (r * C8 + c8) * 8);
                vg[q] = ld_stream(dy + (r * C8 + c8) * 8);
            }
        }
        float d = 0.f, s = 0.f;
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const int64_t c8 = lane + 32 * q;
            if (c8 < C8) {
                float a[8], g[8];
                unpack8(vx[q], a);
                unpack8(vg[q], g);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    d = fmaf(g[e], a[e], d);
                    s = fmaf(a[e], a[e], s);
                }
            }
        }
        d = warp_sum(d);
        float rho;
        if (rstd) {
            rho = __ldg(rstd + r);
        } else {
            s = warp_sum(s);
            rho = rsqrtf(s * inv_cols + eps);
        }
        const float k2 = rho * rho * rho * d * inv_cols;
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const int64_t c8 = lane + 32 * q;
            if (c8 < C8) {
                float a[8], g[8], o[8];
                unpack8(vx[q], a);
                unpack8(vg[q], g);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = rho * g[e] - k2 * a[e];
                st_stream(dx + (r * C8 + c8) * 8, pack8(o));
            }
        }
    }
}

template <int R>
__global__ void __launch_bounds__(256)
    k_rms_fwd(const bf16 *__restrict__ x, bf16 *__restrict__ y, float *__restrict__ rstd,
              int64_t rows, int64_t C8, float inv_cols, float eps)
{
    pdl_wait();
    __shared__ float red[8];
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        uint4 v[R];
        float s = 0.f;
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const int64_t c8 = threadIdx.x + int64_t(q) * blockDim.x;
            if (c8 < C8) {
                v[q] = ld_stream(x + (r * C8 + c8) * 8);
                float f[8];
                unpack8(v[q], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) s = fmaf(f[e], f[e], s);
            }
        }
        s = block_sum(s, red);
        const float rho = rsqrtf(s * inv_cols + eps);
        if (rstd && threadIdx.x == 0) rstd[r] = rho;
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const int64_t c8 = threadIdx.x + int64_t(q) * blockDim.x;
            if (c8 < C8) {
                float f[8];
                unpack8(v[q], f);
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] *= rho;
                st_stream(y + (r * C8 + c8) * 8, pack8(f));
            }
        }
    }
}

template <int R>
__global__ void __launch_bounds__(256)
    k_rms_bwd(const bf16 *__restrict__ dy, const bf16 *__restrict__ x,
              const float *__restrict__ rstd, bf16 *__restrict__ dx, int64_t rows, int64_t C8,
              float inv_cols, float eps)
{
    pdl_wait();
    __shared__ float red[8];
    for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
        uint4 vx[R], vg[R];
        float d = 0.f, s = 0.f;
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const int64_t c8 = threadIdx.x + int64_t(q) * blockDim.x;
            if (c8 < C8) {
                vx[q] = ld_stream(x + (r * C8 + c8) * 8);
                vg[q] = ld_stream(dy + (r * C8 + c8) * 8);
                float a[8], g[8];
                unpack8(vx[q], a);
                unpack8(vg[q], g);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    d = fmaf(g[e], a[e], d);
                    s = fmaf(a[e], a[e], s);
                }
            }
        }
        d = block_sum(d, red);
        float rho;
        if (rstd) {
            rho = __ldg(rstd + r);
        } else {
            s = block_sum(s, red);
            rho = rsqrtf(s * inv_cols + eps);
        }
        const float k2 = rho * rho * rho * d * inv_cols;
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const int64_t c8 = threadIdx.x + int64_t(q) * blockDim.x;
            if (c8 < C8) {
                float a[8], g[8], o[8];
                unpack8(vx[q], a);
                unpack8(vg[q], g);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[e] = rho * g[e] - k2 * a[e];
                st_stream(dx + (r * C8 + c8) * 8, pack8(o));
            }
        }
    }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
cudaError_t launch_aggregate_fwd(const bf16 *x, const float *Hpre, bf16 *y, int64_t T, int n,
                                 int64_t C, cudaStream_t s, bool per_token)
{
    const int64_t C8 = C / 8;
    const unsigned g = grid_for(T, 8);
    const int th = threads_for(C8);
    MHC_PROF("k_agg_fwd", s);
    if (n == 4) {
        if (per_token)
            launch_k(k_agg_fwd<4, false>, dim3(g), dim3(th), 0, s, x, Hpre, y, T, C8);
        else
            launch_k(k_agg_fwd<4, true>, dim3(g), dim3(th), 0, s, x, Hpre, y, T, C8);
    } else {
        if (per_token)
            launch_k(k_agg_fwd<8, false>, dim3(g), dim3(th), 0, s, x, Hpre, y, T, C8);
        else
            launch_k(k_agg_fwd<8, true>, dim3(g), dim3(th), 0, s, x, Hpre, y, T, C8);
    }
    return cudaGetLastError();
}

int agg_static_blocks(int64_t T)
{
    const int64_t want = (T + 7) / 8, cap = int64_t(kSplitSms) * 8;
    return int(want < cap ? (want > 0 ? want : 1) : cap);
}

size_t agg_static_ws_bytes(int64_t T, int n) { return ws_align(size_t(agg_static_blocks(T)) * n * 4); }

cudaError_t launch_aggregate_bwd_static(const bf16 *dy, const bf16 *x, const float *Hpre,
                                        bf16 *dx, float *dHpre, int64_t T, int n, int64_t C,
                                        void *ws, cudaStream_t s)
{
    const int64_t C8 = C / 8;
    const int nb = agg_static_blocks(T);
    float *part = static_cast<float *>(ws);
    {
        MHC_PROF("k_agg_bwd_static", s);
        if (n == 4)
            launch_k(k_agg_bwd_static<4>, dim3(unsigned(nb)), dim3(256), 0, s, dy, x, Hpre, dx, part, T, C8);
        else
            launch_k(k_agg_bwd_static<8>, dim3(unsigned(nb)), dim3(256), 0, s, dy, x, Hpre, dx, part, T, C8);
    }
    {
        MHC_PROF("k_col_sum", s);
        launch_k(k_col_sum, dim3(1), dim3(dim3(32, 32)), 0, s, part, nb, n, dHpre);
    }
    return cudaGetLastError();
}

cudaError_t launch_aggregate_bwd(const bf16 *dy, const bf16 *x, const float *Hpre, bf16 *dx,
                                 float *dHpre, int64_t T, int n, int64_t C, cudaStream_t s)
{
    const int64_t C8 = C / 8;
    const unsigned g = grid_for((T + 7) / 8, 8);
    if (n == 4) {
        MHC_PROF("k_agg_bwd", s);
        launch_k(k_agg_bwd<4>, dim3(g), dim3(256), 0, s, dy, x, Hpre, dx, dHpre, T, C8);
    } else {
        MHC_PROF("k_agg_bwd", s);
        launch_k(k_agg_bwd<8>, dim3(g), dim3(256), 0, s, dy, x, Hpre, dx, dHpre, T, C8);
    }
    return cudaGetLastError();
}

cudaError_t launch_post_fwd(const bf16 *res, const bf16 *f, const bf16 *bias, const float *Hres,
                            const float *Hpost, bf16 *out, int64_t T, int n, int64_t C,
                            cudaStream_t s)
{
    const int64_t C8 = C / 8;
    const unsigned g = grid_for((T + 7) / 8, 8);
    if (n == 4) {
        MHC_PROF("k_post_fwd", s);
        launch_k(k_post_fwd<4>, dim3(g), dim3(256), 0, s, res, f, bias, Hres, Hpost, out, T, C8);
    } else {
        MHC_PROF("k_post_fwd", s);
        launch_k(k_post_fwd8<1>, dim3(grid_for((T + 3) / 4, 16)), dim3(128), 0, s, res, f, bias,
                 Hres, Hpost, out, T, C8);
    }
    return cudaGetLastError();
}

cudaError_t launch_post_bwd_tok(const bf16 *dout, const bf16 *res, const bf16 *f,
                                const bf16 *bias, const float *Hres, const float *Hpost,
                                bf16 *dres, bf16 *df, float *dHres, float *dHpost, int64_t T,
                                int n, int64_t C, cudaStream_t s)
{
    const int64_t C8 = C / 8;
    const unsigned g = grid_for((T + 7) / 8, 8);
    if (n == 4) {
        MHC_PROF("k_post_bwd_tok", s);
        launch_k(k_post_bwd_tok<4>, dim3(g), dim3(256), 0, s, dout, res, f, bias, Hres, Hpost, dres, df, dHres,
                                            dHpost, T, C8);
    } else {
        MHC_PROF("k_post_bwd_tok", s);
        launch_k(k_post_bwd_tok<8>, dim3(g), dim3(256), 0, s, dout, res, f, bias, Hres, Hpost, dres, df, dHres,
                                            dHpost, T, C8);
    }
    return cudaGetLastError();
}

// rows of up to 256 threads x R chunks x 8 values
static int rms_R(int64_t C8)
{
    if (C8 <= 256 * 4) return 4;
    if (C8 <= 256 * 16) return 16;
    return 0;
}

cudaError_t launch_rms_fwd(const bf16 *x, bf16 *y, float *rstd, int64_t rows, int64_t cols,
                           float eps, cudaStream_t s)
{
    const int64_t C8 = cols / 8;
    const float ic = 1.0f / float(cols);
    if (C8 <= 32 * 16) {
        const unsigned g = grid_for((rows + 7) / 8, 8);
        if (C8 <= 32 * 4) {
            MHC_PROF("k_rms_fwd", s);
            launch_k(k_rms_fwd_w<4>, dim3(g), dim3(256), 0, s, x, y, rstd, rows, C8, ic, eps);
        } else if (C8 <= 32 * 8) {
            MHC_PROF("k_rms_fwd", s);
            launch_k(k_rms_fwd_w<8>, dim3(g), dim3(256), 0, s, x, y, rstd, rows, C8, ic, eps);
        } else {
            MHC_PROF("k_rms_fwd", s);
            launch_k(k_rms_fwd_w<16>, dim3(g), dim3(256), 0, s, x, y, rstd, rows, C8, ic, eps);
        }
        return cudaGetLastError();
    }
    const unsigned g = grid_for(rows, 8);
    if (rms_R(C8) == 4) {
        MHC_PROF("k_rms_fwd", s);
        launch_k(k_rms_fwd<4>, dim3(g), dim3(threads_for((C8 + 3) / 4)), 0, s, x, y, rstd, rows, C8, ic, eps);
    } else {
        MHC_PROF("k_rms_fwd", s);
        launch_k(k_rms_fwd<16>, dim3(g), dim3(256), 0, s, x, y, rstd, rows, C8, ic, eps);
    }
    return cudaGetLastError();
}

cudaError_t launch_rms_bwd(const bf16 *dy, const bf16 *x, const float *rstd, bf16 *dx,
                           int64_t rows, int64_t cols, float eps, cudaStream_t s)
{
    const int64_t C8 = cols / 8;
    const float ic = 1.0f / float(cols);
    if (C8 <= 32 * 16) {
        const unsigned g = grid_for((rows + 7) / 8, 8);
        if (C8 <= 32 * 4) {
            MHC_PROF("k_rms_bwd", s);
            launch_k(k_rms_bwd_w<4>, dim3(g), dim3(256), 0, s, dy, x, rstd, dx, rows, C8, ic, eps);
        } else if (C8 <= 32 * 8) {
            MHC_PROF("k_rms_bwd", s);
            launch_k(k_rms_bwd_w<8>, dim3(g), dim3(256), 0, s, dy, x, rstd, dx, rows, C8, ic, eps);
        } else {
            MHC_PROF("k_rms_bwd", s);
            launch_k(k_rms_bwd_w<16>, dim3(g), dim3(256), 0, s, dy, x, rstd, dx, rows, C8, ic, eps);
        }
        return cudaGetLastError();
    }
    const unsigned g = grid_for(rows, 8);
    if (rms_R(C8) == 4) {
        MHC_PROF("k_rms_bwd", s);
        launch_k(k_rms_bwd<4>, dim3(g), dim3(threads_for((C8 + 3) / 4)), 0, s, dy, x, rstd, dx, rows, C8, ic, eps);
    } else {
        MHC_PROF("k_rms_bwd", s);
        launch_k(k_rms_bwd<16>, dim3(g), dim3(256), 0, s, dy, x, rstd, dx, rows, C8, ic, eps);
    }
    return cudaGetLastError();
}

}  // namespace mhc
