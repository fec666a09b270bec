// proj_rms_compute_h forward for callers that cannot allocate device memory.
//
// Some callers cannot hand the library a workspace: an allocator-free
// runtime with no device heap, a plugin that is not allowed to own device
// memory, or a latency-critical path that must not call cudaMalloc/cudaFree
// (which can synchronise the whole device).  For them this file keeps the
// forward's scratch in a fixed array in device global memory that is part
// of the library image itself.  The array
// exists on every GPU that loads the library and stays there until the
// process exits, so its size is kept modest (kNoAllocScratchBytes).
//
// In host code the array's name is only a host-side handle, not a device
// address, so its device address is looked up with cudaGetSymbolAddress
// once per device (with that device current) and cached.  The first call on
// a device does that lookup; make that first call before any stream capture.
// The cache is per device index and holds the address in the context that
// was current at that first call (the device's primary context, for CUDA
// runtime users): it is not valid after cudaDeviceReset or in another
// context on the same device.  Threads may make their first calls
// concurrently (the slots are atomic; both lookups give the same address).
//
// Every call on a device uses the same array.  The kernels overwrite each
// scratch element before they read it, so nothing needs clearing between
// calls, but two calls whose work overlaps on the GPU (different streams,
// no ordering between them) race on the array and give wrong results.
#include <stdio.h>

#include <atomic>

#include "../../include/mhc.h"
#include "launch.h"

namespace {

constexpr size_t kNoAllocScratchBytes = MHC_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

void *scratch_for_current_device(cudaError_t *err)
{
    static std::atomic<void *> ptrs[64];
    int dev = 0;
    *err = cudaGetDevice(&dev);
    if (*err != cudaSuccess) return nullptr;
    if (dev < 0 || dev >= 64) {
        *err = cudaErrorInvalidDevice;
        return nullptr;
    }
    void *p = ptrs[dev].load(std::memory_order_acquire);
    if (!p) {
        *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (*err != cudaSuccess) return nullptr;
        ptrs[dev].store(p, std::memory_order_release);
    }
    return p;
}

}  // namespace

extern "C" {

mhc_status mhc_proj_rms_compute_h_fwd_noalloc(const mhc_bf16 *x, const float *W,
                                              const float *alpha3, const float *b, int64_t T,
                                              int n, int64_t C, int iters, float eps_sk,
                                              float eps_rms, float *H_pre, float *H_post,
                                              float *H_res, float *u_save, float *r_save,
                                              mhc_stream_t stream)
{
    // Same argument rules as mhc_proj_rms_compute_h_fwd; the scratch size
    // that call would need must fit in the fixed array.
    if (T < 0 || (n != 4 && n != 8) || C < 8 || C % 8 != 0)
        return mhc_proj_rms_compute_h_fwd(x, W, alpha3, b, T, n, C, iters, eps_sk, eps_rms,
                                          H_pre, H_post, H_res, u_save, r_save, nullptr, 0,
                                          stream);
    const size_t need = mhc::proj_fwd_ws_bytes(T, n, C);
    if (need > kNoAllocScratchBytes) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "mhc_proj_rms_compute_h_fwd_noalloc: T=%lld n=%d C=%lld needs %zu bytes of "
                 "scratch, more than the fixed %zu",
                 (long long)T, n, (long long)C, need, kNoAllocScratchBytes);
        mhc::set_error_message(msg);
        return MHC_ERR_WORKSPACE_TOO_SMALL;
    }
    if (T == 0)
        return mhc_proj_rms_compute_h_fwd(x, W, alpha3, b, T, n, C, iters, eps_sk, eps_rms,
                                          H_pre, H_post, H_res, u_save, r_save, nullptr, 0,
                                          stream);
    cudaError_t e = cudaSuccess;
    void *scratch = scratch_for_current_device(&e);
    if (!scratch) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "mhc_proj_rms_compute_h_fwd_noalloc: scratch address lookup failed (%s)",
                 cudaGetErrorString(e));
        mhc::set_error_message(msg);
        cudaGetLastError();
        return e == cudaErrorNoDevice ? MHC_ERR_NO_DEVICE : MHC_ERR_CUDA;
    }
    return mhc_proj_rms_compute_h_fwd(x, W, alpha3, b, T, n, C, iters, eps_sk, eps_rms, H_pre,
                                      H_post, H_res, u_save, r_save, scratch,
                                      kNoAllocScratchBytes, stream);
}

}  // extern "C"
