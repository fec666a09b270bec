"""The allocation-free forward entry point.

mhc_proj_rms_compute_h_fwd_noalloc serves callers that cannot allocate a
device workspace (allocator-free runtimes, plugins that may not own device
memory, paths that must not call cudaMalloc/cudaFree).  It takes its scratch
from a fixed array inside the library and runs the same kernels, in the same
order, as the workspace-taking entry point, so its outputs must be bitwise
equal to that entry point's.  Here it is called through the C ABI twice in a
row on different inputs (and once through the Python wrapper), including the
largest documented case and the batch-invariant mode; sizes beyond the fixed
scratch are rejected on the host.  This file is collected last so that a run
stopping at the first failure has already run every other test.
"""
import ctypes

import pytest
import torch

import mhc_inputs as mi
from tests._util import dev_bf16, dev_f32

pytestmark = pytest.mark.gpu

ITERS, EPS = 20, 1e-6
OP_FWD = 1  # MHC_OP_PROJ_RMS_COMPUTE_H_FWD
SCRATCH = 8 << 20  # MHC_NOALLOC_SCRATCH_BYTES


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from layers_proj_rms_gb300 import build
    build.build()
    import layers_proj_rms_gb300 as m
    return m


def _outs(T, n):
    O = n * n + 2 * n
    return [torch.empty(T, n, device="cuda"), torch.empty(T, n, device="cuda"),
            torch.empty(T, n, n, device="cuda"), torch.empty(T, O, device="cuda"),
            torch.empty(T, device="cuda")]


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _same(ref, got):
    for r, g in zip(ref, got):
        assert torch.isfinite(g).all()
        assert torch.equal(r, g), "the allocation-free call differs from the workspace call"


def _run_pair(L, T, n, C, seed, alpha, b_std):
    lib = L.lib
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    inp = mi.layer_inputs(T, n, C, seed, alpha=alpha, b_std=b_std, grads=False)
    x, W = dev_bf16(inp["x"]), dev_f32(inp["W"])
    a, b = dev_f32(inp["alpha"]), dev_f32(inp["b"])
    ref, got = _outs(T, n), _outs(T, n)
    ws = L.workspace(L.OP_PROJ_RMS_COMPUTE_H_FWD, T, n, C)
    st = lib.mhc_proj_rms_compute_h_fwd(_p(x), _p(W), _p(a), _p(b), T, n, C, ITERS,
                                        ctypes.c_float(EPS), ctypes.c_float(EPS),
                                        *[_p(t) for t in ref], _p(ws),
                                        ctypes.c_size_t(ws.numel()), stream)
    assert st == 0, lib.mhc_last_error()
    st = lib.mhc_proj_rms_compute_h_fwd_noalloc(_p(x), _p(W), _p(a), _p(b), T, n, C, ITERS,
                                                ctypes.c_float(EPS), ctypes.c_float(EPS),
                                                *[_p(t) for t in got], stream)
    assert st == 0, lib.mhc_last_error()
    torch.cuda.synchronize()
    _same(ref, got)


# (16384, 4, 4096) is the 7B-scale forward, the largest case the header
# documents as fitting the fixed scratch.
@pytest.mark.parametrize("T,n,C", [(256, 4, 256), (1000, 4, 4096), (300, 8, 1024),
                                   (16384, 4, 4096)])
def test_noalloc_matches_workspace_entry_point_twice(L, T, n, C):
    assert L.lib.mhc_workspace_bytes(OP_FWD, T, n, C) <= SCRATCH
    for call, seed in enumerate((21, 22)):
        _run_pair(L, T, n, C, seed + T, alpha=1.0 if call else 0.01, b_std=0.5 if call else 0.0)


def test_noalloc_batch_invariant_mode(L):
    """The mode changes the K splits and with them the scratch size: a case
    that fits is bitwise equal to the workspace call, the 7B-scale one no
    longer fits and is rejected."""
    L.mhc_set_batch_invariant(True)
    try:
        _run_pair(L, 8192, 4, 4096, 31, alpha=1.0, b_std=0.5)
        T, n, C = 16384, 4, 4096
        assert L.lib.mhc_workspace_bytes(OP_FWD, T, n, C) > SCRATCH
        x = torch.empty(T, n, C, dtype=torch.bfloat16, device="cuda")
        W = torch.empty(n * C, n * n + 2 * n, device="cuda")
        a, b = torch.empty(3, device="cuda"), torch.empty(n * n + 2 * n, device="cuda")
        with pytest.raises(Exception, match="scratch"):
            L.mhc_proj_rms_compute_h_fwd_noalloc(x, W, a, b, ITERS, EPS, EPS, *_outs(T, n))
    finally:
        L.mhc_set_batch_invariant(False)


def test_noalloc_python_wrapper(L):
    """The binding's wrapper of the entry point gives the same bits."""
    T, n, C = 512, 4, 1024
    inp = mi.layer_inputs(T, n, C, 41, alpha=1.0, b_std=0.5, grads=False)
    x, W = dev_bf16(inp["x"]), dev_f32(inp["W"])
    a, b = dev_f32(inp["alpha"]), dev_f32(inp["b"])
    ref, got = _outs(T, n), _outs(T, n)
    L.mhc_proj_rms_compute_h_fwd(x, W, a, b, ITERS, EPS, EPS, *ref,
                                 L.workspace(L.OP_PROJ_RMS_COMPUTE_H_FWD, T, n, C))
    L.mhc_proj_rms_compute_h_fwd_noalloc(x, W, a, b, ITERS, EPS, EPS, *got)
    torch.cuda.synchronize()
    _same(ref, got)


def test_noalloc_rejects_sizes_beyond_its_scratch(L):
    lib = L.lib
    T, n, C = 1 << 20, 8, 7168
    need = lib.mhc_workspace_bytes(OP_FWD, T, n, C)
    assert need > SCRATCH
    A = ctypes.c_void_p(0x10000)
    st = lib.mhc_proj_rms_compute_h_fwd_noalloc(A, A, A, A, T, n, C, ITERS, ctypes.c_float(EPS),
                                                ctypes.c_float(EPS), A, A, A, None, None, None)
    assert st == 5
    assert b"scratch" in lib.mhc_last_error()
