// Batched Sinkhorn-Knopp forward and backward: one launch for all M
// matrices (rwkv-ops mhu_ffi.cu SinkhornFwdHost/SinkhornBwdHost run one
// launch per matrix from a host loop).  n = 4: one thread per matrix, the
// 16 entries in registers; n = 8: each lane owns one row and a group of n
// lanes owns one matrix.
#include "launch.h"
#include "sinkhorn.cuh"

namespace mhc {

constexpr int kSkThreads = 128;

template <int N>
__device__ __forceinline__ void load_row(const float *p, float (&v)[N])
{
    const float4 *q = reinterpret_cast<const float4 *>(p);
#pragma unroll
    for (int h = 0; h < N / 4; ++h) {
        const float4 w = __ldg(q + h);
        v[4 * h] = w.x;
        v[4 * h + 1] = w.y;
        v[4 * h + 2] = w.z;
        v[4 * h + 3] = w.w;
    }
}

template <int N>
__device__ __forceinline__ void store_row(float *p, const float (&v)[N])
{
    float4 *q = reinterpret_cast<float4 *>(p);
#pragma unroll
    for (int h = 0; h < N / 4; ++h)
        q[h] = make_float4(v[4 * h], v[4 * h + 1], v[4 * h + 2], v[4 * h + 3]);
}

template <int N>
__global__ void __launch_bounds__(kSkThreads)
    k_sinkhorn_fwd(const float *__restrict__ logits, float *__restrict__ P, int64_t rows,
                   int iters, float eps)
{
    pdl_wait();
    const int64_t row = int64_t(blockIdx.x) * kSkThreads + threadIdx.x;  // = m*N + i
    const bool live = row < rows;
    float a[N];
    if (live) {
        load_row<N>(logits + row * N, a);
#pragma unroll
        for (int j = 0; j < N; ++j) a[j] = expf(a[j]);
    } else {
#pragma unroll
        for (int j = 0; j < N; ++j) a[j] = 1.f;
    }
    sk_forward<N>(a, iters, eps, nullptr, 0);
    if (live) store_row<N>(P + row * N, a);
}

template <int N>
__global__ void __launch_bounds__(kSkThreads)
    k_sinkhorn_bwd(const float *__restrict__ dP, const float *__restrict__ logits,
                   float *__restrict__ dlogits, int64_t rows, int iters, float eps)
{
    pdl_wait();
    extern __shared__ float sk_store[];  // [2*iters][kSkThreads]
    const int64_t row = int64_t(blockIdx.x) * kSkThreads + threadIdx.x;
    const bool live = row < rows;
    float a[N], e[N], g[N];
    if (live) {
        load_row<N>(logits + row * N, e);
        load_row<N>(dP + row * N, g);
#pragma unroll
        for (int j = 0; j < N; ++j) e[j] = expf(e[j]);
    } else {
#pragma unroll
        for (int j = 0; j < N; ++j) {
            e[j] = 1.f;
            g[j] = 0.f;
        }
    }
#pragma unroll
    for (int j = 0; j < N; ++j) a[j] = e[j];
    float *store = sk_store + threadIdx.x;
    sk_forward<N>(a, iters, eps, store, kSkThreads);
    sk_backward<N>(g, a, e, iters, store, kSkThreads);
    if (live) store_row<N>(dlogits + row * N, g);
}

// n = 4, one thread per matrix (sk4_forward / sk4_backward); the backward
// keeps the denominators in shared memory, thread-major.
constexpr int kSk1Threads = 64;

__device__ __forceinline__ void sk1_load(const float *p, float (&m)[4][4])
{
    const float4 *q = reinterpret_cast<const float4 *>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 w = __ldg(q + i);
        m[i][0] = w.x;
        m[i][1] = w.y;
        m[i][2] = w.z;
        m[i][3] = w.w;
    }
}

__device__ __forceinline__ void sk1_store(float *p, const float (&m)[4][4])
{
    float4 *q = reinterpret_cast<float4 *>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) q[i] = make_float4(m[i][0], m[i][1], m[i][2], m[i][3]);
}

__global__ void __launch_bounds__(kSk1Threads)
    k_sinkhorn1_fwd(const float *__restrict__ logits, float *__restrict__ P, int64_t M, int iters,
                    float eps)
{
    pdl_wait();
    const int64_t m = int64_t(blockIdx.x) * kSk1Threads + threadIdx.x;
    if (m >= M) return;
    float a[4][4];
    sk1_load(logits + m * 16, a);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) a[i][j] = expf(a[i][j]);
    sk4_forward(a, iters, eps, nullptr, 0);
    sk1_store(P + m * 16, a);
}

__global__ void __launch_bounds__(kSk1Threads)
    k_sinkhorn1_bwd(const float *__restrict__ dP, const float *__restrict__ logits,
                    float *__restrict__ dlogits, int64_t M, int iters, float eps)
{
    pdl_wait();
    extern __shared__ float sk1_st[];   // [8 iters][kSk1Threads]
    const int64_t m = int64_t(blockIdx.x) * kSk1Threads + threadIdx.x;
    if (m >= M) return;
    float e[4][4], a[4][4], g[4][4];
    sk1_load(logits + m * 16, e);
    sk1_load(dP + m * 16, g);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) a[i][j] = e[i][j] = expf(e[i][j]);
    float *store = sk1_st + threadIdx.x;
    sk4_forward(a, iters, eps, store, kSk1Threads);
    sk4_backward(g, a, e, iters, store, kSk1Threads);
    sk1_store(dlogits + m * 16, g);
}

static size_t sk1_smem(int iters) { return size_t(8) * iters * kSk1Threads * sizeof(float); }

static size_t sk_smem(int iters) { return size_t(2) * iters * kSkThreads * sizeof(float); }

cudaError_t launch_sinkhorn_fwd(const float *logits, float *P, int64_t M, int n, int iters,
                                float eps, cudaStream_t s)
{
    const int64_t rows = M * n;
    const unsigned grid = unsigned((rows + kSkThreads - 1) / kSkThreads);
    if (n == 4) {
        MHC_PROF("k_sinkhorn_fwd", s);
        launch_k(k_sinkhorn1_fwd, dim3(unsigned((M + kSk1Threads - 1) / kSk1Threads)),
                 dim3(kSk1Threads), 0, s, logits, P, M, iters, eps);
    } else {
        MHC_PROF("k_sinkhorn_fwd", s);
        launch_k(k_sinkhorn_fwd<8>, dim3(grid), dim3(kSkThreads), 0, s, logits, P, rows, iters, eps);
    }
    return cudaGetLastError();
}

cudaError_t launch_sinkhorn_bwd(const float *dP, const float *logits, float *dlogits, int64_t M,
                                int n, int iters, float eps, cudaStream_t s)
{
    const int64_t rows = M * n;
    const unsigned grid = unsigned((rows + kSkThreads - 1) / kSkThreads);
    const size_t smem = sk_smem(iters);
    cudaError_t e;
    if (n == 4) {
        e = set_smem_limit(reinterpret_cast<const void *>(k_sinkhorn1_bwd), int(sk1_smem(64)));
        if (e != cudaSuccess) return e;
        {
            MHC_PROF("k_sinkhorn_bwd", s);
            launch_k(k_sinkhorn1_bwd, dim3(unsigned((M + kSk1Threads - 1) / kSk1Threads)),
                     dim3(kSk1Threads), sk1_smem(iters), s, dP, logits, dlogits, M, iters, eps);
        }
    } else {
        e = set_smem_limit(reinterpret_cast<const void *>(k_sinkhorn_bwd<8>), int(sk_smem(64)));
        if (e != cudaSuccess) return e;
        {
            MHC_PROF("k_sinkhorn_bwd", s);
            launch_k(k_sinkhorn_bwd<8>, dim3(grid), dim3(kSkThreads), smem, s, dP, logits, dlogits, rows, iters, eps);
        }
    }
    return cudaGetLastError();
}

}  // namespace mhc
