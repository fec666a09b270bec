// The C ABI of libmhc (declared in include/mhc.h): host-side validation,
// status codes, workspace sizing and dispatch to the kernel launchers.
// Nothing here allocates device memory.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <nvtx3/nvToolsExt.h>

#include "../../include/mhc.h"
#include "launch.h"

using mhc::bf16;

namespace {

thread_local char g_msg[512] = "";

mhc_status fail(mhc_status st, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return st;
}

// The device-side fault word (see mhc_device_error).
__device__ int g_fault_word;

int *fault_ptr()
{
    static int *ptrs[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!ptrs[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_fault_word) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<int *>(p);
    }
    return ptrs[dev];
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Host-side argument checks of one entry point.  Its lifetime is the call's:
// it also brackets the call in an NVTX range named after the entry point (no
// cost unless a profiler is attached).
struct Check {
    mhc_status st = MHC_OK;
    const char *fn;
    explicit Check(const char *f) : fn(f)
    {
        g_msg[0] = '\0';
        nvtxRangePushA(f);
    }
    ~Check() { nvtxRangePop(); }
    Check(const Check &) = delete;
    Check &operator=(const Check &) = delete;

    Check &ptr(const void *p, const char *name)
    {
        if (st == MHC_OK && !p) st = fail(MHC_ERR_NULL_PTR, "%s: %s is NULL", fn, name);
        if (st == MHC_OK && p && !aligned16(p))
            st = fail(MHC_ERR_MISALIGNED, "%s: %s is not 16-byte aligned", fn, name);
        return *this;
    }
    Check &opt(const void *p, const char *name)  // may be NULL
    {
        if (st == MHC_OK && p && !aligned16(p))
            st = fail(MHC_ERR_MISALIGNED, "%s: %s is not 16-byte aligned", fn, name);
        return *this;
    }
    Check &count(int64_t v, const char *name)
    {
        if (st == MHC_OK && v < 0) st = fail(MHC_ERR_BAD_SHAPE, "%s: %s = %lld < 0", fn, name, (long long)v);
        return *this;
    }
    Check &nstreams(int n)
    {
        if (st == MHC_OK && n != 4 && n != 8)
            st = fail(MHC_ERR_UNSUPPORTED_N, "%s: n = %d (supported: 4, 8)", fn, n);
        return *this;
    }
    Check &channels(int64_t C, const char *name = "C")
    {
        if (st == MHC_OK && (C < 8 || C % 8 != 0))
            st = fail(MHC_ERR_BAD_SHAPE, "%s: %s = %lld must be a positive multiple of 8", fn, name,
                      (long long)C);
        if (st == MHC_OK && C > (int64_t(1) << 30))
            st = fail(MHC_ERR_BAD_SHAPE, "%s: %s = %lld too large", fn, name, (long long)C);
        return *this;
    }
    // the tensor-core kernels address rows and the flattened k = i*C + c with
    // 32-bit TMA coordinates
    Check &tma(int64_t T, int64_t K)
    {
        if (st == MHC_OK && (T > INT32_MAX || K > INT32_MAX))
            st = fail(MHC_ERR_BAD_SHAPE, "%s: T = %lld and n*C = %lld must be below 2^31", fn,
                      (long long)T, (long long)K);
        return *this;
    }
    Check &fits(int64_t a, int64_t b, const char *what)  // a*b elements must fit in int64 / 2^62
    {
        if (st == MHC_OK && a > 0 && b > 0 && a > (int64_t(1) << 62) / b)
            st = fail(MHC_ERR_BAD_SHAPE, "%s: %s overflows", fn, what);
        return *this;
    }
    Check &iters(int it)
    {
        if (st == MHC_OK && (it < 0 || it > MHC_MAX_ITERS))
            st = fail(MHC_ERR_BAD_ARG, "%s: iters = %d outside [0, %d]", fn, it, MHC_MAX_ITERS);
        return *this;
    }
    Check &eps(float e, const char *name)
    {
        if (st == MHC_OK && !(e >= 0.f && isfinite(e)))
            st = fail(MHC_ERR_BAD_ARG, "%s: %s = %g must be finite and >= 0", fn, name, double(e));
        return *this;
    }
    Check &ws(const void *p, size_t have, size_t need)
    {
        if (st == MHC_OK && have < need)
            st = fail(MHC_ERR_WORKSPACE_TOO_SMALL, "%s: workspace %zu bytes < %zu needed", fn, have,
                      need);
        if (st == MHC_OK && need > 0 && !p)
            st = fail(MHC_ERR_NULL_PTR, "%s: workspace is NULL", fn);
        if (st == MHC_OK && p && (reinterpret_cast<uintptr_t>(p) & 255u))
            st = fail(MHC_ERR_MISALIGNED, "%s: workspace is not 256-byte aligned", fn);
        return *this;
    }
    Check &device()
    {
        if (st != MHC_OK) return *this;
        int dev = -1;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) {
            cudaGetLastError();
            st = fail(MHC_ERR_NO_DEVICE, "%s: no CUDA device (%s)", fn, cudaGetErrorString(e));
        }
        return *this;
    }
};

mhc_status launched(const char *fn, cudaError_t e)
{
    if (e != cudaSuccess)
        return fail(MHC_ERR_CUDA, "%s: CUDA error %s (%s)", fn, cudaGetErrorName(e),
                    cudaGetErrorString(e));
    return MHC_OK;
}

size_t layer_fwd_ws(int64_t T, int n, int64_t C) { return mhc::proj_fwd_ws_bytes(T, n, C); }

// With no tokens every sum over tokens is zero.
mhc_status zero_param_grads(Check &ck, float *dW, int64_t nW, float *dalpha, float *db,
                            int64_t nb, float *dbias, int64_t nbias, cudaStream_t s)
{
    if (ck.device().st) return ck.st;
    cudaError_t e = cudaMemsetAsync(dW, 0, size_t(nW) * sizeof(float), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dalpha, 0, 3 * sizeof(float), s);
    if (e == cudaSuccess) e = cudaMemsetAsync(db, 0, size_t(nb) * sizeof(float), s);
    if (e == cudaSuccess && dbias) e = cudaMemsetAsync(dbias, 0, size_t(nbias) * sizeof(float), s);
    return launched(ck.fn, e);
}

// Bit-reproducible mode: its reduction trees are defined for four streams.
mhc_status pinned_n4(Check &ck, int n)
{
    if (ck.st == MHC_OK && n != 4)
        ck.st = fail(MHC_ERR_UNSUPPORTED_N,
                     "%s: the pinned-reduction mode is defined for n = 4 (got n = %d)", ck.fn, n);
    return ck.st;
}

// backward workspaces cover the pinned mode's per-token scratch too
size_t proj_bwd_ws(int64_t T, int n, int64_t C)
{
    const size_t a = mhc::proj_bwd_ws_bytes(T, n, C), b = n == 4 ? mhc::pin_bwd_ws_bytes(T) : 0;
    return a > b ? a : b;
}

}  // namespace

void mhc::set_error_message(const char *msg) { snprintf(g_msg, sizeof g_msg, "%s", msg); }

extern "C" {

const char *mhc_status_string(mhc_status s)
{
    switch (s) {
    case MHC_OK: return "ok";
    case MHC_ERR_NULL_PTR: return "null pointer";
    case MHC_ERR_BAD_SHAPE: return "bad shape";
    case MHC_ERR_MISALIGNED: return "misaligned pointer";
    case MHC_ERR_UNSUPPORTED_N: return "unsupported number of streams";
    case MHC_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MHC_ERR_BAD_ARG: return "bad argument";
    case MHC_ERR_CUDA: return "CUDA error";
    case MHC_ERR_NO_DEVICE: return "no CUDA device";
    case MHC_ERR_DEVICE_FAULT: return "device-side fault reported";
    }
    return "unknown status";
}

const char *mhc_last_error(void) { return g_msg; }

int mhc_version(void) { return 100; }

void mhc_set_batch_invariant(int on) { mhc::set_batch_invariant(on); }

void mhc_set_pinned_reductions(int on) { mhc::set_pinned(on); }

int mhc_pinned_reductions(void) { return mhc::pinned(); }

int mhc_batch_invariant(void) { return mhc::batch_invariant(); }

mhc_status mhc_selftest_wait_timeout(int wait_us, mhc_stream_t stream)
{
    Check ck("mhc_selftest_wait_timeout");
    if (wait_us < 1 || wait_us > 1000000)
        return fail(MHC_ERR_BAD_SHAPE, "mhc_selftest_wait_timeout: wait_us must be in [1, 1e6]");
    if (ck.device().st) return ck.st;
    int dev = 0, khz = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev);
    if (e != cudaSuccess) return launched(ck.fn, e);
    const long long cycles = (long long)wait_us * (khz > 0 ? khz : 2000000) / 1000;
    return launched(ck.fn, mhc::launch_selftest_wait(cycles, fault_ptr(), stream));
}

mhc_status mhc_device_error(int *code, mhc_stream_t stream)
{
    Check ck("mhc_device_error");
    if (ck.device().st) return ck.st;
    int *p = fault_ptr();
    if (!p) return fail(MHC_ERR_CUDA, "mhc_device_error: fault word unavailable");
    int v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, p, sizeof v, cudaMemcpyDeviceToHost, stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    if (e == cudaSuccess && v != 0) {
        const int zero = 0;
        e = cudaMemcpyAsync(p, &zero, sizeof zero, cudaMemcpyHostToDevice, stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
    }
    if (e != cudaSuccess) return launched("mhc_device_error", e);
    if (code) *code = v;
    if (v != 0) return fail(MHC_ERR_DEVICE_FAULT, "a kernel reported fault code %d", v);
    return MHC_OK;
}

size_t mhc_workspace_bytes(mhc_op op, int64_t T, int n, int64_t C)
{
    if (T < 0 || C < 8 || C % 8 != 0) return 0;
    if (op == MHC_OP_RMSNORM_RESIDUAL_BWD) return mhc::norm_ws_bytes(T, C);  // n unused
    if (n != 4 && n != 8) return 0;
    switch (op) {
    case MHC_OP_RMSNORM_RESIDUAL_BWD: return 0;
    case MHC_OP_H_AGGREGATE_RMSNORM_BWD: return mhc::norm_ws_bytes(T, C);
    case MHC_OP_H_AGGREGATE_STATIC_BWD: return mhc::agg_static_ws_bytes(T, n);
    case MHC_OP_PROJ_RMS_PARTIAL_FWD: return mhc::proj_fwd_ws_bytes(T, n, C);
    case MHC_OP_COMPUTE_H_BWD: return mhc::compute_h_bwd_ws_bytes(T, n);
    case MHC_OP_PROJ_RMS_PARTIAL_BWD: return mhc::proj_bwd_ws_bytes(T, n, C);
    case MHC_OP_PROJ_RMS_COMPUTE_H_FWD: return mhc::proj_fwd_ws_bytes(T, n, C);
    case MHC_OP_PROJ_RMS_COMPUTE_H_BWD: return proj_bwd_ws(T, n, C);
    case MHC_OP_H_POST_BDA_BWD: return mhc::dbias_ws_bytes(T, C);
    case MHC_OP_LAYER_FWD: return layer_fwd_ws(T, n, C);
    case MHC_OP_LAYER_BWD: return proj_bwd_ws(T, n, C);
    case MHC_OP_H_POST_BDA_COMPUTE_H_FWD: return mhc::post_proj_ws_bytes(T, n, C);
    }
    return 0;
}

mhc_status mhc_sinkhorn_fwd(const float *logits, float *P, int64_t M, int n, int iters,
                            float eps, mhc_stream_t stream)
{
    Check ck("mhc_sinkhorn_fwd");
    ck.count(M, "M").nstreams(n).fits(M, n * n, "M*n*n").iters(iters).eps(eps, "eps");
    if (ck.st || M == 0) return ck.st;
    ck.ptr(logits, "logits").ptr(P, "P");
    if (ck.st) return ck.st;
    if (ck.device().st) return ck.st;
    if (mhc::pinned())
        return pinned_n4(ck, n) ? ck.st
                                : launched(ck.fn, mhc::launch_pin_sinkhorn_fwd(logits, P, M, iters,
                                                                               eps, stream));
    return launched(ck.fn, mhc::launch_sinkhorn_fwd(logits, P, M, n, iters, eps, stream));
}

mhc_status mhc_sinkhorn_bwd(const float *dP, const float *logits, float *dlogits, int64_t M,
                            int n, int iters, float eps, mhc_stream_t stream)
{
    Check ck("mhc_sinkhorn_bwd");
    ck.count(M, "M").nstreams(n).fits(M, n * n, "M*n*n").iters(iters).eps(eps, "eps");
    if (ck.st || M == 0) return ck.st;
    ck.ptr(dP, "dP").ptr(logits, "logits").ptr(dlogits, "dlogits");
    if (ck.st) return ck.st;
    if (ck.device().st) return ck.st;
    if (mhc::pinned())
        return pinned_n4(ck, n) ? ck.st
                                : launched(ck.fn, mhc::launch_pin_sinkhorn_bwd(dP, logits, dlogits,
                                                                               M, iters, eps, stream));
    return launched(ck.fn, mhc::launch_sinkhorn_bwd(dP, logits, dlogits, M, n, iters, eps, stream));
}

mhc_status mhc_proj_rms_compute_h_fwd(const mhc_bf16 *x, const float *W, const float *alpha3,
                                      const float *b, int64_t T, int n, int64_t C, int iters,
                                      float eps_sk, float eps_rms, float *H_pre, float *H_post,
                                      float *H_res, float *u_save, float *r_save, void *ws,
                                      size_t ws_bytes, mhc_stream_t stream)
{
    Check ck("mhc_proj_rms_compute_h_fwd");
    ck.count(T, "T").nstreams(n).channels(C).fits(T, n * C, "T*n*C").tma(T, n * C).iters(iters);
    ck.eps(eps_sk, "eps_sk").eps(eps_rms, "eps_rms");
    if (ck.st || T == 0) return ck.st;
    ck.ptr(x, "x").ptr(W, "W").ptr(alpha3, "alpha3").ptr(b, "b").ptr(H_pre, "H_pre");
    ck.ptr(H_post, "H_post").ptr(H_res, "H_res").opt(u_save, "u_save").opt(r_save, "r_save");
    ck.ws(ws, ws_bytes, mhc::proj_fwd_ws_bytes(T, n, C)).device();
    if (ck.st) return ck.st;
    if (mhc::pinned())
        return pinned_n4(ck, n) ? ck.st
                                : launched(ck.fn, mhc::launch_pin_proj_fwd(
                                                      reinterpret_cast<const bf16 *>(x), W, alpha3,
                                                      b, T, C, iters, eps_sk, eps_rms, H_pre,
                                                      H_post, H_res, u_save, r_save, stream));
    return launched(ck.fn, mhc::launch_proj_fwd(reinterpret_cast<const bf16 *>(x), W, alpha3, b,
                                                T, n, C, iters, eps_sk, eps_rms, H_pre, H_post,
                                                H_res, u_save, r_save, ws, fault_ptr(), stream));
}

mhc_status mhc_proj_rms_compute_h_bwd(const float *dH_pre, const float *dH_post,
                                      const float *dH_res, const mhc_bf16 *x, const float *W,
                                      const float *alpha3, const float *b, const float *u_save,
                                      const float *r_save, int64_t T, int n, int64_t C,
                                      int iters, float eps_sk, float eps_rms, mhc_bf16 *dx,
                                      float *dW, float *dalpha3, float *db, void *ws,
                                      size_t ws_bytes, mhc_stream_t stream)
{
    Check ck("mhc_proj_rms_compute_h_bwd");
    ck.count(T, "T").nstreams(n).channels(C).fits(T, n * C, "T*n*C").tma(T, n * C).iters(iters);
    ck.eps(eps_sk, "eps_sk").eps(eps_rms, "eps_rms");
    ck.ptr(W, "W").ptr(alpha3, "alpha3").ptr(b, "b").ptr(dW, "dW").ptr(dalpha3, "dalpha3");
    ck.ptr(db, "db");
    if (ck.st) return ck.st;
    if (T == 0) return zero_param_grads(ck, dW, int64_t(n) * C * (n * n + 2 * n), dalpha3, db,
                                        n * n + 2 * n, nullptr, 0, stream);
    ck.ptr(dH_pre, "dH_pre").ptr(dH_post, "dH_post").ptr(dH_res, "dH_res").ptr(x, "x");
    ck.ptr(u_save, "u_save").ptr(r_save, "r_save").ptr(dx, "dx");
    ck.ws(ws, ws_bytes, proj_bwd_ws(T, n, C)).device();
    if (ck.st) return ck.st;
    if (mhc::pinned())
        return pinned_n4(ck, n) ? ck.st
                                : launched(ck.fn, mhc::launch_pin_proj_bwd(
                                                      dH_pre, dH_post, dH_res,
                                                      reinterpret_cast<const bf16 *>(x), W, alpha3,
                                                      b, T, C, iters, eps_sk, eps_rms,
                                                      reinterpret_cast<bf16 *>(dx), dW, dalpha3, db,
                                                      ws, stream));
    return launched(ck.fn, mhc::launch_proj_bwd(dH_pre, dH_post, dH_res,
                                                reinterpret_cast<const bf16 *>(x), W, alpha3, b,
                                                u_save, r_save, T, n, C, iters, eps_sk, eps_rms,
                                                reinterpret_cast<bf16 *>(dx), dW, dalpha3, db, ws,
                                                fault_ptr(), stream));
}

mhc_status mhc_h_aggregate_fwd(const mhc_bf16 *x, const float *H_pre, mhc_bf16 *y, int64_t T,
                               int n, int64_t C, mhc_stream_t stream)
{
    Check ck("mhc_h_aggregate_fwd");
    ck.count(T, "T").nstreams(n).channels(C).fits(T, n * C, "T*n*C");
    if (ck.st || T == 0) return ck.st;
    ck.ptr(x, "x").ptr(H_pre, "H_pre").ptr(y, "y");
    if (ck.st) return ck.st;
    if (ck.device().st) return ck.st;
    if (mhc::pinned())
        return pinned_n4(ck, n) ? ck.st
                                : launched(ck.fn, mhc::launch_pin_agg_fwd(
                                                      reinterpret_cast<const bf16 *>(x), H_pre,
                                                      reinterpret_cast<bf16 *>(y), T, C, stream));
    return launched(ck.fn, mhc::launch_aggregate_fwd(reinterpret_cast<const bf16 *>(x), H_pre,
                                                     reinterpret_cast<bf16 *>(y), T, n, C, stream));
}

mhc_status mhc_h_aggregate_bwd(const mhc_bf16 *dy, const mhc_bf16 *x, const float *H_pre,
                               mhc_bf16 *dx, float *dH_pre, int64_t T, int n, int64_t C,
                               mhc_stream_t stream)
{
    Check ck("mhc_h_aggregate_bwd");
    ck.count(T, "T").nstreams(n).channels(C).fits(T, n * C, "T*n*C");
    if (ck.st || T == 0) return ck.st;
    ck.ptr(dy, "dy").ptr(x, "x").ptr(H_pre, "H_pre").ptr(dx, "dx").ptr(dH_pre, "dH_pre");
    if (ck.st) return ck.st;
    if (ck.device().st) return ck.st;
    if (mhc::pinned())
        return pinned_n4(ck, n) ? ck.st
                                : launched(ck.fn, mhc::launch_pin_agg_bwd(
                                                      reinterpret_cast<const bf16 *>(dy),
                                                      reinterpret_cast<const bf16 *>(x), H_pre,
                                                      reinterpret_cast<bf16 *>(dx), dH_pre, T, C,
                                                      stream));
    return launched(ck.fn, mhc::launch_aggregate_bwd(
                               reinterpret_cast<const bf16 *>(dy), reinterpret_cast<const bf16 *>(x),
                               H_pre, reinterpret_cast<bf16 *>(dx), dH_pre, T, n, C, stream));
}

mhc_status mhc_h_post_bda_fwd(const mhc_bf16 *residual, const mhc_bf16 *f, const mhc_bf16 *bias,
                              const float *H_res, const float *H_post, mhc_bf16 *out, int64_t T,
                              int n, int64_t C, mhc_stream_t stream)
{
    Check ck("mhc_h_post_bda_fwd");
    ck.count(T, "T").nstreams(n).channels(C).fits(T, n * C, "T*n*C");
    if (ck.st || T == 0) return ck.st;
    ck.ptr(residual, "residual").ptr(f, "f").opt(bias, "bias").ptr(H_res, "H_res");
    ck.ptr(H_post, "H_post").ptr(out, "out");
    if (ck.st) return ck.st;
    if (ck.device().st) return ck.st;
    if (mhc::pinned())
        return pinned_n4(ck, n) ? ck.st
                                : launched(ck.fn, mhc::launch_pin_post_fwd(
                                                      reinterpret_cast<const bf16 *>(residual),
                                                      reinterpret_cast<const bf16 *>(f),
                                                      reinterpret_cast<const bf16 *>(bias), H_res,
                                                      H_post, reinterpret_cast<bf16 *>(out), T, C,
                                                      stream));
    return launched(ck.fn, mhc::launch_post_fwd(reinterpret_cast<const bf16 *>(residual),
                                                reinterpret_cast<const bf16 *>(f),
                                                reinterpret_cast<const bf16 *>(bias), H_res, H_post,
                                                reinterpret_cast<bf16 *>(out), T, n, C, stream));
}

mhc_status mhc_h_post_bda_compute_h_fwd(
    const mhc_bf16 *residual, const mhc_bf16 *f, const mhc_bf16 *bias, const float *H_res,
    const float *H_post, const float *W_next, const float *alpha3_next, const float *b_next,
    int64_t T, int n, int64_t C, int iters, float eps_sk, float eps_rms, mhc_bf16 *out,
    float *H_pre_next, float *H_post_next, float *H_res_next, float *u_save_next,
    float *r_save_next, void *ws, size_t ws_bytes, mhc_stream_t stream)
{
    Check ck("mhc_h_post_bda_compute_h_fwd");
    ck.count(T, "T").nstreams(n).channels(C).fits(T, n * C, "T*n*C").tma(T, n * C).iters(iters);
    ck.eps(eps_sk, "eps_sk").eps(eps_rms, "eps_rms");
    if (ck.st || T == 0) return ck.st;
    ck.ptr(residual, "residual").ptr(f, "f").opt(bias, "bias").ptr(H_res, "H_res");
    ck.ptr(H_post, "H_post").ptr(W_next, "W_next").ptr(alpha3_next, "alpha3_next");
    ck.ptr(b_next, "b_next").ptr(out, "out").ptr(H_pre_next, "H_pre_next");
    ck.ptr(H_post_next, "H_post_next").ptr(H_res_next, "H_res_next");
    ck.opt(u_save_next, "u_save_next").opt(r_save_next, "r_save_next");
    ck.ws(ws, ws_bytes, mhc::post_proj_ws_bytes(T, n, C)).device();
    if (ck.st) return ck.st;
    return launched(ck.fn, mhc::launch_post_proj_fwd(
                               reinterpret_cast<const bf16 *>(residual),
                               reinterpret_cast<const bf16 *>(f), reinterpret_cast<const bf16 *>(bias),
                               H_res, H_post, W_next, alpha3_next, b_next, T, n, C, iters, eps_sk,
                               eps_rms, reinterpret_cast<bf16 *>(out), H_pre_next, H_post_next,
                               H_res_next, u_save_next, r_save_next, ws, fault_ptr(), stream));
}

mhc_status mhc_h_post_bda_bwd(const mhc_bf16 *dout, const mhc_bf16 *residual, const mhc_bf16 *f,
                              const mhc_bf16 *bias, const float *H_res, const float *H_post,
                              mhc_bf16 *dresidual, mhc_bf16 *df, float *dbias, float *dH_res,
                              float *dH_post, int64_t T, int n, int64_t C, void *ws,
                              size_t ws_bytes, mhc_stream_t stream)
{
    Check ck("mhc_h_post_bda_bwd");
    ck.count(T, "T").nstreams(n).channels(C).fits(T, n * C, "T*n*C").opt(dbias, "dbias");
    if (ck.st) return ck.st;
    if (T == 0) {
        if (dbias) {  // an empty sum is zero
            if (ck.device().st) return ck.st;
            return launched(ck.fn, cudaMemsetAsync(dbias, 0, size_t(C) * sizeof(float), stream));
        }
        return MHC_OK;
    }
    ck.ptr(dout, "dout").ptr(residual, "residual").ptr(f, "f").opt(bias, "bias");
    ck.ptr(H_res, "H_res").ptr(H_post, "H_post").ptr(dresidual, "dresidual").ptr(df, "df");
    ck.ptr(dH_res, "dH_res").ptr(dH_post, "dH_post");
    ck.ws(ws, ws_bytes, dbias ? mhc::dbias_ws_bytes(T, C) : 0).device();
    if (ck.st) return ck.st;
    const bf16 *g = reinterpret_cast<const bf16 *>(dout);
    if (mhc::pinned())
        return pinned_n4(ck, n) ? ck.st
                                : launched(ck.fn, mhc::launch_pin_post_bwd(
                                                      g, reinterpret_cast<const bf16 *>(residual),
                                                      reinterpret_cast<const bf16 *>(f),
                                                      reinterpret_cast<const bf16 *>(bias), H_res,
                                                      H_post, reinterpret_cast<bf16 *>(dresidual),
                                                      reinterpret_cast<bf16 *>(df), dbias, dH_res,
                                                      dH_post, T, C, stream));
    cudaError_t e = mhc::launch_post_bwd_tok(
        g, reinterpret_cast<const bf16 *>(residual), reinterpret_cast<const bf16 *>(f),
        reinterpret_cast<const bf16 *>(bias), H_res, H_post, reinterpret_cast<bf16 *>(dresidual),
        reinterpret_cast<bf16 *>(df), dH_res, dH_post, T, n, C, stream);
    if (e == cudaSuccess && dbias) e = mhc::launch_dbias(g, H_post, dbias, T, n, C, ws, stream);
    return launched(ck.fn, e);
}

static int64_t kMaxRmsCols = 32768;

mhc_status rmsnorm_fwd(const mhc_bf16 *x, mhc_bf16 *y, float *rstd, int64_t rows, int64_t cols,
                       float eps, mhc_stream_t stream)
{
    Check ck("rmsnorm_fwd");
    ck.count(rows, "rows").channels(cols, "cols").fits(rows, cols, "rows*cols").eps(eps, "eps");
    if (ck.st == MHC_OK && cols > kMaxRmsCols)
        ck.st = fail(MHC_ERR_BAD_SHAPE, "rmsnorm_fwd: cols = %lld > %lld", (long long)cols,
                     (long long)kMaxRmsCols);
    if (ck.st || rows == 0) return ck.st;
    ck.ptr(x, "x").ptr(y, "y").opt(rstd, "rstd").device();
    if (ck.st) return ck.st;
    return launched(ck.fn, mhc::launch_rms_fwd(reinterpret_cast<const bf16 *>(x),
                                               reinterpret_cast<bf16 *>(y), rstd, rows, cols, eps,
                                               stream));
}

mhc_status rmsnorm_bwd(const mhc_bf16 *dy, const mhc_bf16 *x, const float *rstd, mhc_bf16 *dx,
                       int64_t rows, int64_t cols, float eps, mhc_stream_t stream)
{
    Check ck("rmsnorm_bwd");
    ck.count(rows, "rows").channels(cols, "cols").fits(rows, cols, "rows*cols").eps(eps, "eps");
    if (ck.st == MHC_OK && cols > kMaxRmsCols)
        ck.st = fail(MHC_ERR_BAD_SHAPE, "rmsnorm_bwd: cols = %lld > %lld", (long long)cols,
                     (long long)kMaxRmsCols);
    if (ck.st || rows == 0) return ck.st;
    ck.ptr(dy, "dy").ptr(x, "x").opt(rstd, "rstd").ptr(dx, "dx").device();
    if (ck.st) return ck.st;
    return launched(ck.fn, mhc::launch_rms_bwd(reinterpret_cast<const bf16 *>(dy),
                                               reinterpret_cast<const bf16 *>(x), rstd,
                                               reinterpret_cast<bf16 *>(dx), rows, cols, eps,
                                               stream));
}

mhc_status mhc_layer_fwd(const mhc_bf16 *x, const float *W, const float *alpha3, const float *b,
                         const mhc_bf16 *f, const mhc_bf16 *bias, int64_t T, int n, int64_t C,
                         int iters, float eps_sk, float eps_rms, float *H_pre, float *H_post,
                         float *H_res, float *u_save, float *r_save, mhc_bf16 *y,
                         mhc_bf16 *out, void *ws, size_t ws_bytes, mhc_stream_t stream)
{
    Check ck("mhc_layer_fwd");
    ck.count(T, "T").nstreams(n).channels(C).fits(T, n * C, "T*n*C").tma(T, n * C).iters(iters);
    ck.eps(eps_sk, "eps_sk").eps(eps_rms, "eps_rms");
    if (ck.st || T == 0) return ck.st;
    ck.ptr(x, "x").ptr(W, "W").ptr(alpha3, "alpha3").ptr(b, "b").ptr(f, "f").opt(bias, "bias");
    ck.ptr(H_pre, "H_pre").ptr(H_post, "H_post").ptr(H_res, "H_res").ptr(u_save, "u_save");
    ck.ptr(r_save, "r_save").ptr(y, "y").ptr(out, "out");
    ck.ws(ws, ws_bytes, layer_fwd_ws(T, n, C)).device();
    if (ck.st) return ck.st;
    const bf16 *xb = reinterpret_cast<const bf16 *>(x);
    if (mhc::pinned())
        return pinned_n4(ck, n) ? ck.st
                                : launched(ck.fn, mhc::launch_pin_layer_fwd(
                                                      xb, W, alpha3, b,
                                                      reinterpret_cast<const bf16 *>(f),
                                                      reinterpret_cast<const bf16 *>(bias), T, C,
                                                      iters, eps_sk, eps_rms, H_pre, H_post, H_res,
                                                      u_save, r_save, reinterpret_cast<bf16 *>(y),
                                                      reinterpret_cast<bf16 *>(out), stream));
    cudaError_t e = mhc::launch_proj_fwd(xb, W, alpha3, b, T, n, C, iters, eps_sk, eps_rms, H_pre,
                                         H_post, H_res, u_save, r_save, ws, fault_ptr(), stream);
    if (e == cudaSuccess)
        e = mhc::launch_aggregate_fwd(xb, H_pre, reinterpret_cast<bf16 *>(y), T, n, C, stream);
    if (e == cudaSuccess)
        e = mhc::launch_post_fwd(xb, reinterpret_cast<const bf16 *>(f),
                                 reinterpret_cast<const bf16 *>(bias), H_res, H_post,
                                 reinterpret_cast<bf16 *>(out), T, n, C, stream);
    return launched(ck.fn, e);
}

mhc_status mhc_layer_bwd(const mhc_bf16 *dout, const mhc_bf16 *dy, const mhc_bf16 *x,
                         const float *W, const float *alpha3, const float *b, const mhc_bf16 *f,
                         const mhc_bf16 *bias, const float *H_pre, const float *H_post,
                         const float *H_res, const float *u_save, const float *r_save,
                         int64_t T, int n, int64_t C, int iters, float eps_sk, float eps_rms,
                         mhc_bf16 *dx, mhc_bf16 *df, float *dW, float *dalpha3, float *db,
                         float *dbias, void *ws, size_t ws_bytes, mhc_stream_t stream)
{
    Check ck("mhc_layer_bwd");
    ck.count(T, "T").nstreams(n).channels(C).fits(T, n * C, "T*n*C").tma(T, n * C).iters(iters);
    ck.eps(eps_sk, "eps_sk").eps(eps_rms, "eps_rms");
    ck.ptr(W, "W").ptr(alpha3, "alpha3").ptr(b, "b").opt(bias, "bias").ptr(dW, "dW");
    ck.ptr(dalpha3, "dalpha3").ptr(db, "db").opt(dbias, "dbias");
    if (ck.st == MHC_OK && bias && !dbias)
        ck.st = fail(MHC_ERR_NULL_PTR, "mhc_layer_bwd: dbias is NULL but bias is given");
    if (ck.st) return ck.st;
    if (T == 0) return zero_param_grads(ck, dW, int64_t(n) * C * (n * n + 2 * n), dalpha3, db,
                                        n * n + 2 * n, dbias, C, stream);
    ck.ptr(dout, "dout").ptr(dy, "dy").ptr(x, "x").ptr(f, "f").ptr(H_pre, "H_pre");
    ck.ptr(H_post, "H_post").ptr(H_res, "H_res").ptr(u_save, "u_save").ptr(r_save, "r_save");
    ck.ptr(dx, "dx").ptr(df, "df");
    ck.ws(ws, ws_bytes, proj_bwd_ws(T, n, C)).device();
    if (ck.st) return ck.st;
    if (mhc::pinned())
        return pinned_n4(ck, n) ? ck.st
                                : launched(ck.fn, mhc::launch_pin_layer_bwd(
                                                      reinterpret_cast<const bf16 *>(dout),
                                                      reinterpret_cast<const bf16 *>(dy),
                                                      reinterpret_cast<const bf16 *>(x), W, alpha3,
                                                      b, reinterpret_cast<const bf16 *>(f),
                                                      reinterpret_cast<const bf16 *>(bias), H_pre,
                                                      H_post, H_res, T, C, iters, eps_sk, eps_rms,
                                                      reinterpret_cast<bf16 *>(dx),
                                                      reinterpret_cast<bf16 *>(df), dW, dalpha3, db,
                                                      dbias, ws, stream));
    return launched(
        ck.fn, mhc::launch_layer_bwd(reinterpret_cast<const bf16 *>(dout),
                                     reinterpret_cast<const bf16 *>(dy),
                                     reinterpret_cast<const bf16 *>(x), W, alpha3, b,
                                     reinterpret_cast<const bf16 *>(f),
                                     reinterpret_cast<const bf16 *>(bias), H_pre, H_post, H_res,
                                     u_save, r_save, T, n, C, iters, eps_sk, eps_rms,
                                     reinterpret_cast<bf16 *>(dx), reinterpret_cast<bf16 *>(df),
                                     dW, dalpha3, db, dbias, ws, fault_ptr(), stream));
}

/* ---------------------------------------------------------------------- */
/* Ops beyond the layer path                                               */
/* ---------------------------------------------------------------------- */

mhc_status mhc_h_aggregate_static_fwd(const mhc_bf16 *x, const float *H_pre, mhc_bf16 *y,
                                      int64_t T, int n, int64_t C, mhc_stream_t stream)
{
    Check ck("mhc_h_aggregate_static_fwd");
    ck.count(T, "T").nstreams(n).channels(C).fits(T, n * C, "T*n*C");
    if (ck.st || T == 0) return ck.st;
    ck.ptr(x, "x").ptr(H_pre, "H_pre").ptr(y, "y").device();
    if (ck.st) return ck.st;
    return launched(ck.fn, mhc::launch_aggregate_fwd(reinterpret_cast<const bf16 *>(x), H_pre,
                                                     reinterpret_cast<bf16 *>(y), T, n, C, stream,
                                                     false));
}

mhc_status mhc_h_aggregate_static_bwd(const mhc_bf16 *dy, const mhc_bf16 *x, const float *H_pre,
                                      mhc_bf16 *dx, float *dH_pre, int64_t T, int n, int64_t C,
                                      void *ws, size_t ws_bytes, mhc_stream_t stream)
{
    Check ck("mhc_h_aggregate_static_bwd");
    ck.count(T, "T").nstreams(n).channels(C).fits(T, n * C, "T*n*C");
    ck.ptr(H_pre, "H_pre").ptr(dH_pre, "dH_pre");
    if (ck.st) return ck.st;
    if (T == 0) {
        if (ck.device().st) return ck.st;
        return launched(ck.fn, cudaMemsetAsync(dH_pre, 0, size_t(n) * sizeof(float), stream));
    }
    ck.ptr(dy, "dy").ptr(x, "x").opt(dx, "dx");
    ck.ws(ws, ws_bytes, mhc::agg_static_ws_bytes(T, n)).device();
    if (ck.st) return ck.st;
    return launched(ck.fn, mhc::launch_aggregate_bwd_static(
                               reinterpret_cast<const bf16 *>(dy), reinterpret_cast<const bf16 *>(x),
                               H_pre, reinterpret_cast<bf16 *>(dx), dH_pre, T, n, C, ws, stream));
}

mhc_status rmsnorm_residual_fwd(const mhc_bf16 *x, const mhc_bf16 *res, const float *gamma,
                                mhc_bf16 *h, mhc_bf16 *y, float *rstd, int64_t rows,
                                int64_t cols, float eps, mhc_stream_t stream)
{
    Check ck("rmsnorm_residual_fwd");
    ck.count(rows, "rows").channels(cols, "cols").fits(rows, cols, "rows*cols").eps(eps, "eps");
    if (ck.st == MHC_OK && cols > kMaxRmsCols)
        ck.st = fail(MHC_ERR_BAD_SHAPE, "rmsnorm_residual_fwd: cols = %lld > %lld",
                     (long long)cols, (long long)kMaxRmsCols);
    if (ck.st || rows == 0) return ck.st;
    ck.ptr(x, "x").opt(res, "res").opt(gamma, "gamma").opt(h, "h").ptr(y, "y").opt(rstd, "rstd");
    if (ck.device().st) return ck.st;
    return launched(ck.fn, mhc::launch_rmsr_fwd(reinterpret_cast<const bf16 *>(x),
                                                reinterpret_cast<const bf16 *>(res), gamma,
                                                reinterpret_cast<bf16 *>(h),
                                                reinterpret_cast<bf16 *>(y), rstd, rows, cols,
                                                eps, stream));
}

mhc_status rmsnorm_residual_bwd(const mhc_bf16 *dy, const mhc_bf16 *dh, const mhc_bf16 *x,
                                const mhc_bf16 *res, const float *gamma, const float *rstd,
                                mhc_bf16 *dx, float *dgamma, int64_t rows, int64_t cols,
                                float eps, void *ws, size_t ws_bytes, mhc_stream_t stream)
{
    Check ck("rmsnorm_residual_bwd");
    ck.count(rows, "rows").channels(cols, "cols").fits(rows, cols, "rows*cols").eps(eps, "eps");
    if (ck.st == MHC_OK && cols > kMaxRmsCols)
        ck.st = fail(MHC_ERR_BAD_SHAPE, "rmsnorm_residual_bwd: cols = %lld > %lld",
                     (long long)cols, (long long)kMaxRmsCols);
    ck.opt(dgamma, "dgamma");
    if (ck.st) return ck.st;
    if (rows == 0) {
        if (!dgamma || ck.device().st) return ck.st;
        return launched(ck.fn, cudaMemsetAsync(dgamma, 0, size_t(cols) * sizeof(float), stream));
    }
    ck.ptr(dy, "dy").opt(dh, "dh").ptr(x, "x").opt(res, "res").opt(gamma, "gamma");
    ck.opt(rstd, "rstd").ptr(dx, "dx");
    if (dgamma) ck.ws(ws, ws_bytes, mhc::norm_ws_bytes(rows, cols));
    if (ck.device().st) return ck.st;
    return launched(ck.fn, mhc::launch_rmsr_bwd(
                               reinterpret_cast<const bf16 *>(dy), reinterpret_cast<const bf16 *>(dh),
                               reinterpret_cast<const bf16 *>(x), reinterpret_cast<const bf16 *>(res),
                               gamma, rstd, reinterpret_cast<bf16 *>(dx), dgamma, rows, cols, eps,
                               ws, stream));
}

mhc_status mhc_h_aggregate_rmsnorm_fwd(const mhc_bf16 *x, const float *H_pre, const float *gamma,
                                       mhc_bf16 *y, mhc_bf16 *yn, float *rstd, int64_t T, int n,
                                       int64_t C, float eps, mhc_stream_t stream)
{
    Check ck("mhc_h_aggregate_rmsnorm_fwd");
    ck.count(T, "T").nstreams(n).channels(C).fits(T, n * C, "T*n*C").eps(eps, "eps");
    if (ck.st == MHC_OK && C > kMaxRmsCols)
        ck.st = fail(MHC_ERR_BAD_SHAPE, "mhc_h_aggregate_rmsnorm_fwd: C = %lld > %lld",
                     (long long)C, (long long)kMaxRmsCols);
    if (ck.st || T == 0) return ck.st;
    ck.ptr(x, "x").ptr(H_pre, "H_pre").opt(gamma, "gamma").opt(y, "y").ptr(yn, "yn");
    ck.opt(rstd, "rstd");
    if (ck.device().st) return ck.st;
    return launched(ck.fn, mhc::launch_aggn_fwd(reinterpret_cast<const bf16 *>(x), H_pre, gamma,
                                                reinterpret_cast<bf16 *>(y),
                                                reinterpret_cast<bf16 *>(yn), rstd, T, n, C, eps,
                                                stream));
}

mhc_status mhc_h_aggregate_rmsnorm_bwd(const mhc_bf16 *dyn, const mhc_bf16 *dy, const mhc_bf16 *x,
                                       const float *H_pre, const float *gamma, const float *rstd,
                                       mhc_bf16 *dx, float *dH_pre, float *dgamma, int64_t T,
                                       int n, int64_t C, float eps, void *ws, size_t ws_bytes,
                                       mhc_stream_t stream)
{
    Check ck("mhc_h_aggregate_rmsnorm_bwd");
    ck.count(T, "T").nstreams(n).channels(C).fits(T, n * C, "T*n*C").eps(eps, "eps");
    if (ck.st == MHC_OK && C > kMaxRmsCols)
        ck.st = fail(MHC_ERR_BAD_SHAPE, "mhc_h_aggregate_rmsnorm_bwd: C = %lld > %lld",
                     (long long)C, (long long)kMaxRmsCols);
    ck.opt(dgamma, "dgamma");
    if (ck.st) return ck.st;
    if (T == 0) {
        if (!dgamma || ck.device().st) return ck.st;
        return launched(ck.fn, cudaMemsetAsync(dgamma, 0, size_t(C) * sizeof(float), stream));
    }
    ck.ptr(dyn, "dyn").opt(dy, "dy").ptr(x, "x").ptr(H_pre, "H_pre").opt(gamma, "gamma");
    ck.opt(rstd, "rstd").ptr(dx, "dx").ptr(dH_pre, "dH_pre");
    if (dgamma) ck.ws(ws, ws_bytes, mhc::norm_ws_bytes(T, C));
    if (ck.device().st) return ck.st;
    return launched(ck.fn, mhc::launch_aggn_bwd(
                               reinterpret_cast<const bf16 *>(dyn), reinterpret_cast<const bf16 *>(dy),
                               reinterpret_cast<const bf16 *>(x), H_pre, gamma, rstd,
                               reinterpret_cast<bf16 *>(dx), dH_pre, dgamma, T, n, C, eps, ws,
                               stream));
}

mhc_status mhc_proj_rms_partial_fwd(const mhc_bf16 *x_shard, const float *W_shard, int64_t T,
                                    int n, int64_t Cs, float *u_part, float *s_part, void *ws,
                                    size_t ws_bytes, mhc_stream_t stream)
{
    Check ck("mhc_proj_rms_partial_fwd");
    ck.count(T, "T").nstreams(n).channels(Cs, "Cs").fits(T, n * Cs, "T*n*Cs").tma(T, n * Cs);
    if (ck.st || T == 0) return ck.st;
    ck.ptr(x_shard, "x_shard").ptr(W_shard, "W_shard").ptr(u_part, "u_part").ptr(s_part, "s_part");
    ck.ws(ws, ws_bytes, mhc::proj_fwd_ws_bytes(T, n, Cs)).device();
    if (ck.st) return ck.st;
    return launched(ck.fn, mhc::launch_proj_partial_sums(reinterpret_cast<const bf16 *>(x_shard),
                                                         W_shard, T, n, Cs, u_part, s_part, ws,
                                                         fault_ptr(), stream));
}

mhc_status mhc_compute_h_fwd(const float *u, const float *s, int64_t K, const float *alpha3,
                             const float *b, int64_t T, int n, int iters, float eps_sk,
                             float eps_rms, float *H_pre, float *H_post, float *H_res,
                             float *r_save, mhc_stream_t stream)
{
    Check ck("mhc_compute_h_fwd");
    ck.count(T, "T").nstreams(n).iters(iters).eps(eps_sk, "eps_sk").eps(eps_rms, "eps_rms");
    if (ck.st == MHC_OK && K < 1) ck.st = fail(MHC_ERR_BAD_SHAPE, "mhc_compute_h_fwd: K = %lld < 1", (long long)K);
    if (ck.st || T == 0) return ck.st;
    ck.ptr(u, "u").ptr(s, "s").ptr(alpha3, "alpha3").ptr(b, "b").ptr(H_pre, "H_pre");
    ck.ptr(H_post, "H_post").ptr(H_res, "H_res").opt(r_save, "r_save").device();
    if (ck.st) return ck.st;
    return launched(ck.fn, mhc::launch_compute_h_fwd(u, s, K, alpha3, b, T, n, iters, eps_sk,
                                                     eps_rms, H_pre, H_post, H_res, r_save,
                                                     stream));
}

mhc_status mhc_compute_h_bwd(const float *dH_pre, const float *dH_post, const float *dH_res,
                             const float *u, const float *s, int64_t K, const float *alpha3,
                             const float *b, int64_t T, int n, int iters, float eps_sk,
                             float eps_rms, float *du, float *coef, float *dalpha3, float *db,
                             void *ws, size_t ws_bytes, mhc_stream_t stream)
{
    Check ck("mhc_compute_h_bwd");
    ck.count(T, "T").nstreams(n).iters(iters).eps(eps_sk, "eps_sk").eps(eps_rms, "eps_rms");
    if (ck.st == MHC_OK && K < 1) ck.st = fail(MHC_ERR_BAD_SHAPE, "mhc_compute_h_bwd: K = %lld < 1", (long long)K);
    ck.ptr(dalpha3, "dalpha3").ptr(db, "db");
    if (ck.st) return ck.st;
    if (T == 0) {
        if (ck.device().st) return ck.st;
        cudaError_t e = cudaMemsetAsync(dalpha3, 0, 3 * sizeof(float), stream);
        if (e == cudaSuccess) e = cudaMemsetAsync(db, 0, size_t(n * n + 2 * n) * sizeof(float), stream);
        return launched(ck.fn, e);
    }
    ck.ptr(dH_pre, "dH_pre").ptr(dH_post, "dH_post").ptr(dH_res, "dH_res").ptr(u, "u");
    ck.ptr(s, "s").ptr(alpha3, "alpha3").ptr(b, "b").ptr(du, "du").ptr(coef, "coef");
    ck.ws(ws, ws_bytes, mhc::compute_h_bwd_ws_bytes(T, n)).device();
    if (ck.st) return ck.st;
    return launched(ck.fn, mhc::launch_compute_h_bwd(dH_pre, dH_post, dH_res, u, s, K, alpha3, b,
                                                     T, n, iters, eps_sk, eps_rms, du, coef,
                                                     dalpha3, db, ws, stream));
}

mhc_status mhc_proj_rms_partial_bwd(const mhc_bf16 *x_shard, const float *W_shard,
                                    const float *du, const float *coef, int64_t T, int n,
                                    int64_t Cs, mhc_bf16 *dx_shard, float *dW_shard, void *ws,
                                    size_t ws_bytes, mhc_stream_t stream)
{
    Check ck("mhc_proj_rms_partial_bwd");
    ck.count(T, "T").nstreams(n).channels(Cs, "Cs").fits(T, n * Cs, "T*n*Cs").tma(T, n * Cs);
    ck.ptr(dW_shard, "dW_shard");
    if (ck.st) return ck.st;
    if (T == 0) {
        if (ck.device().st) return ck.st;
        return launched(ck.fn, cudaMemsetAsync(dW_shard, 0,
                                               size_t(n) * Cs * (n * n + 2 * n) * sizeof(float),
                                               stream));
    }
    ck.ptr(x_shard, "x_shard").ptr(W_shard, "W_shard").ptr(du, "du").ptr(coef, "coef");
    ck.ptr(dx_shard, "dx_shard");
    ck.ws(ws, ws_bytes, mhc::proj_bwd_ws_bytes(T, n, Cs)).device();
    if (ck.st) return ck.st;
    return launched(ck.fn, mhc::launch_proj_partial_bwd(
                               reinterpret_cast<const bf16 *>(x_shard), W_shard, du, coef, T, n, Cs,
                               reinterpret_cast<bf16 *>(dx_shard), dW_shard, ws, fault_ptr(),
                               stream));
}

}  // extern "C"
