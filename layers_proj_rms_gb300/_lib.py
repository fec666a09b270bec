"""ctypes marshalling for libmhc (include/mhc.h)."""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "_build", "libmhc.so")

if not os.path.exists(lib_path):
    raise ImportError(
        f"libmhc.so is missing ({lib_path}); build it first with "
        "`python -c 'import __graft_entry__ as g; g.build()'` or "
        "`python -m layers_proj_rms_gb300.build`")

lib = ctypes.CDLL(lib_path)

OP_PROJ_RMS_COMPUTE_H_FWD = 1
OP_PROJ_RMS_COMPUTE_H_BWD = 2
OP_H_POST_BDA_BWD = 3
OP_LAYER_FWD = 4
OP_LAYER_BWD = 5
OP_RMSNORM_RESIDUAL_BWD = 6
OP_H_AGGREGATE_RMSNORM_BWD = 7
OP_H_AGGREGATE_STATIC_BWD = 8
OP_PROJ_RMS_PARTIAL_FWD = 9
OP_COMPUTE_H_BWD = 10
OP_PROJ_RMS_PARTIAL_BWD = 11
OP_H_POST_BDA_COMPUTE_H_FWD = 12

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

_SIGS = {
    "mhc_sinkhorn_fwd": [_P, _P, _I64, _I, _I, _F, _P],
    "mhc_sinkhorn_bwd": [_P, _P, _P, _I64, _I, _I, _F, _P],
    "mhc_proj_rms_compute_h_fwd": [_P, _P, _P, _P, _I64, _I, _I64, _I, _F, _F, _P, _P, _P, _P,
                                   _P, _P, _SZ, _P],
    "mhc_proj_rms_compute_h_bwd": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I, _I64, _I, _F,
                                   _F, _P, _P, _P, _P, _P, _SZ, _P],
    "mhc_h_aggregate_fwd": [_P, _P, _P, _I64, _I, _I64, _P],
    "mhc_h_aggregate_bwd": [_P, _P, _P, _P, _P, _I64, _I, _I64, _P],
    "mhc_h_post_bda_fwd": [_P, _P, _P, _P, _P, _P, _I64, _I, _I64, _P],
    "mhc_h_post_bda_bwd": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I, _I64, _P, _SZ,
                           _P],
    "rmsnorm_fwd": [_P, _P, _P, _I64, _I64, _F, _P],
    "rmsnorm_bwd": [_P, _P, _P, _P, _I64, _I64, _F, _P],
    "mhc_layer_fwd": [_P, _P, _P, _P, _P, _P, _I64, _I, _I64, _I, _F, _F, _P, _P, _P, _P, _P,
                      _P, _P, _P, _SZ, _P],
    "mhc_layer_bwd": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I, _I64, _I, _F,
                      _F, _P, _P, _P, _P, _P, _P, _P, _SZ, _P],
    "mhc_device_error": [ctypes.POINTER(ctypes.c_int), _P],
    "mhc_selftest_wait_timeout": [_I, _P],
    "mhc_proj_rms_compute_h_fwd_noalloc": [_P, _P, _P, _P, _I64, _I, _I64, _I, _F, _F, _P, _P,
                                           _P, _P, _P, _P],
    "mhc_h_aggregate_static_fwd": [_P, _P, _P, _I64, _I, _I64, _P],
    "mhc_h_aggregate_static_bwd": [_P, _P, _P, _P, _P, _I64, _I, _I64, _P, _SZ, _P],
    "rmsnorm_residual_fwd": [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _P],
    "rmsnorm_residual_bwd": [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _F, _P, _SZ, _P],
    "mhc_h_aggregate_rmsnorm_fwd": [_P, _P, _P, _P, _P, _P, _I64, _I, _I64, _F, _P],
    "mhc_h_aggregate_rmsnorm_bwd": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I, _I64, _F, _P,
                                    _SZ, _P],
    "mhc_proj_rms_partial_fwd": [_P, _P, _I64, _I, _I64, _P, _P, _P, _SZ, _P],
    "mhc_compute_h_fwd": [_P, _P, _I64, _P, _P, _I64, _I, _I, _F, _F, _P, _P, _P, _P, _P],
    "mhc_compute_h_bwd": [_P, _P, _P, _P, _P, _I64, _P, _P, _I64, _I, _I, _F, _F, _P, _P, _P, _P,
                          _P, _SZ, _P],
    "mhc_proj_rms_partial_bwd": [_P, _P, _P, _P, _I64, _I, _I64, _P, _P, _P, _SZ, _P],
    "mhc_h_post_bda_compute_h_fwd": [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I, _I64, _I, _F, _F,
                                     _P, _P, _P, _P, _P, _P, _P, _SZ, _P],
}
for _name, _args in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = ctypes.c_int
lib.mhc_status_string.argtypes = [_I]
lib.mhc_status_string.restype = ctypes.c_char_p
lib.mhc_last_error.argtypes = []
lib.mhc_last_error.restype = ctypes.c_char_p
lib.mhc_version.argtypes = []
lib.mhc_version.restype = ctypes.c_int
lib.mhc_set_batch_invariant.argtypes = [_I]
lib.mhc_set_batch_invariant.restype = None
lib.mhc_batch_invariant.argtypes = []
lib.mhc_batch_invariant.restype = ctypes.c_int
lib.mhc_set_pinned_reductions.argtypes = [_I]
lib.mhc_set_pinned_reductions.restype = None
lib.mhc_pinned_reductions.argtypes = []
lib.mhc_pinned_reductions.restype = ctypes.c_int
lib.mhc_workspace_bytes.argtypes = [_I, _I64, _I, _I64]
lib.mhc_workspace_bytes.restype = ctypes.c_size_t


class MhcError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"libmhc status {status} ({lib.mhc_status_string(status).decode()}): "
                         f"{msg}")
        self.status = status


def _ok(st: int) -> None:
    if st != 0:
        raise MhcError(st, lib.mhc_last_error().decode())


def _ptr(t, dtype=None, shape=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() and not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return t.data_ptr() if t.numel() else None


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


_BF, _F32 = torch.bfloat16, torch.float32


def _O(n):
    return n * n + 2 * n


def mhc_version() -> int:
    return int(lib.mhc_version())


def mhc_workspace_bytes(op: int, T: int, n: int, C: int) -> int:
    return int(lib.mhc_workspace_bytes(op, T, n, C))


def workspace(op: int, T: int, n: int, C: int, device=None) -> torch.Tensor:
    """A device buffer of mhc_workspace_bytes(op, T, n, C) bytes (256-aligned)."""
    nb = max(mhc_workspace_bytes(op, T, n, C), 256)
    return torch.empty(nb, dtype=torch.uint8, device=device or "cuda")


def _ws(ws):
    if ws is None:
        return None, 0
    return _ptr(ws, torch.uint8, name="ws"), ws.numel()


def mhc_device_error(stream=None) -> int:
    code = ctypes.c_int(0)
    st = lib.mhc_device_error(ctypes.byref(code), _stream(stream))
    if st not in (0, 9):
        _ok(st)
    return code.value


def mhc_selftest_wait_timeout(wait_us, stream=None):
    _ok(lib.mhc_selftest_wait_timeout(int(wait_us), _stream(stream)))


def mhc_sinkhorn_fwd(logits, P, iters, eps, stream=None):
    n = logits.shape[-1]
    M = logits.numel() // (n * n) if n else 0
    _ok(lib.mhc_sinkhorn_fwd(_ptr(logits, _F32, name="logits"),
                             _ptr(P, _F32, logits.shape, "P"), M, n, iters, eps,
                             _stream(stream)))


def mhc_sinkhorn_bwd(dP, logits, dlogits, iters, eps, stream=None):
    n = logits.shape[-1]
    M = logits.numel() // (n * n) if n else 0
    _ok(lib.mhc_sinkhorn_bwd(_ptr(dP, _F32, logits.shape, "dP"),
                             _ptr(logits, _F32, name="logits"),
                             _ptr(dlogits, _F32, logits.shape, "dlogits"), M, n, iters, eps,
                             _stream(stream)))


def mhc_proj_rms_compute_h_fwd(x, W, alpha3, b, iters, eps_sk, eps_rms, H_pre, H_post, H_res,
                               u_save=None, r_save=None, ws=None, stream=None):
    T, n, C = x.shape
    O = _O(n)
    wp, wb = _ws(ws)
    _ok(lib.mhc_proj_rms_compute_h_fwd(
        _ptr(x, _BF, name="x"), _ptr(W, _F32, (n * C, O), "W"), _ptr(alpha3, _F32, (3,), "alpha3"),
        _ptr(b, _F32, (O,), "b"), T, n, C, iters, eps_sk, eps_rms,
        _ptr(H_pre, _F32, (T, n), "H_pre"), _ptr(H_post, _F32, (T, n), "H_post"),
        _ptr(H_res, _F32, (T, n, n), "H_res"), _ptr(u_save, _F32, (T, O), "u_save"),
        _ptr(r_save, _F32, (T,), "r_save"), wp, wb, _stream(stream)))


def mhc_proj_rms_compute_h_bwd(dH_pre, dH_post, dH_res, x, W, alpha3, b, u_save, r_save, iters,
                               eps_sk, eps_rms, dx, dW, dalpha3, db, ws=None, stream=None):
    T, n, C = x.shape
    O = _O(n)
    wp, wb = _ws(ws)
    _ok(lib.mhc_proj_rms_compute_h_bwd(
        _ptr(dH_pre, _F32, (T, n), "dH_pre"), _ptr(dH_post, _F32, (T, n), "dH_post"),
        _ptr(dH_res, _F32, (T, n, n), "dH_res"), _ptr(x, _BF, name="x"),
        _ptr(W, _F32, (n * C, O), "W"), _ptr(alpha3, _F32, (3,), "alpha3"),
        _ptr(b, _F32, (O,), "b"), _ptr(u_save, _F32, (T, O), "u_save"),
        _ptr(r_save, _F32, (T,), "r_save"), T, n, C, iters, eps_sk, eps_rms,
        _ptr(dx, _BF, (T, n, C), "dx"), _ptr(dW, _F32, (n * C, O), "dW"),
        _ptr(dalpha3, _F32, (3,), "dalpha3"), _ptr(db, _F32, (O,), "db"), wp, wb,
        _stream(stream)))


def mhc_h_aggregate_fwd(x, H_pre, y, stream=None):
    T, n, C = x.shape
    _ok(lib.mhc_h_aggregate_fwd(_ptr(x, _BF, name="x"), _ptr(H_pre, _F32, (T, n), "H_pre"),
                                _ptr(y, _BF, (T, C), "y"), T, n, C, _stream(stream)))


def mhc_h_aggregate_bwd(dy, x, H_pre, dx, dH_pre, stream=None):
    T, n, C = x.shape
    _ok(lib.mhc_h_aggregate_bwd(_ptr(dy, _BF, (T, C), "dy"), _ptr(x, _BF, name="x"),
                                _ptr(H_pre, _F32, (T, n), "H_pre"),
                                _ptr(dx, _BF, (T, n, C), "dx"),
                                _ptr(dH_pre, _F32, (T, n), "dH_pre"), T, n, C, _stream(stream)))


def mhc_h_post_bda_fwd(residual, f, bias, H_res, H_post, out, stream=None):
    T, n, C = residual.shape
    _ok(lib.mhc_h_post_bda_fwd(_ptr(residual, _BF, name="residual"), _ptr(f, _BF, (T, C), "f"),
                               _ptr(bias, _BF, (C,), "bias"),
                               _ptr(H_res, _F32, (T, n, n), "H_res"),
                               _ptr(H_post, _F32, (T, n), "H_post"),
                               _ptr(out, _BF, (T, n, C), "out"), T, n, C, _stream(stream)))


def mhc_h_post_bda_compute_h_fwd(residual, f, bias, H_res, H_post, W_next, alpha3_next, b_next,
                                 iters, eps_sk, eps_rms, out, H_pre_next, H_post_next,
                                 H_res_next, u_save_next=None, r_save_next=None, ws=None,
                                 stream=None):
    T, n, C = residual.shape
    O = _O(n)
    wp, wb = _ws(ws)
    _ok(lib.mhc_h_post_bda_compute_h_fwd(
        _ptr(residual, _BF, name="residual"), _ptr(f, _BF, (T, C), "f"),
        _ptr(bias, _BF, (C,), "bias"), _ptr(H_res, _F32, (T, n, n), "H_res"),
        _ptr(H_post, _F32, (T, n), "H_post"), _ptr(W_next, _F32, (n * C, O), "W_next"),
        _ptr(alpha3_next, _F32, (3,), "alpha3_next"), _ptr(b_next, _F32, (O,), "b_next"),
        T, n, C, iters, eps_sk, eps_rms, _ptr(out, _BF, (T, n, C), "out"),
        _ptr(H_pre_next, _F32, (T, n), "H_pre_next"), _ptr(H_post_next, _F32, (T, n), "H_post_next"),
        _ptr(H_res_next, _F32, (T, n, n), "H_res_next"),
        _ptr(u_save_next, _F32, (T, O), "u_save_next"), _ptr(r_save_next, _F32, (T,), "r_save_next"),
        wp, wb, _stream(stream)))


def mhc_h_post_bda_bwd(dout, residual, f, bias, H_res, H_post, dresidual, df, dbias, dH_res,
                       dH_post, ws=None, stream=None):
    T, n, C = residual.shape
    wp, wb = _ws(ws)
    _ok(lib.mhc_h_post_bda_bwd(
        _ptr(dout, _BF, (T, n, C), "dout"), _ptr(residual, _BF, name="residual"),
        _ptr(f, _BF, (T, C), "f"), _ptr(bias, _BF, (C,), "bias"),
        _ptr(H_res, _F32, (T, n, n), "H_res"), _ptr(H_post, _F32, (T, n), "H_post"),
        _ptr(dresidual, _BF, (T, n, C), "dresidual"), _ptr(df, _BF, (T, C), "df"),
        _ptr(dbias, _F32, (C,), "dbias"), _ptr(dH_res, _F32, (T, n, n), "dH_res"),
        _ptr(dH_post, _F32, (T, n), "dH_post"), T, n, C, wp, wb, _stream(stream)))


def rmsnorm_fwd(x, y, rstd, eps, stream=None):
    rows, cols = x.shape
    _ok(lib.rmsnorm_fwd(_ptr(x, _BF, name="x"), _ptr(y, _BF, (rows, cols), "y"),
                        _ptr(rstd, _F32, (rows,), "rstd"), rows, cols, eps, _stream(stream)))


def rmsnorm_bwd(dy, x, rstd, dx, eps, stream=None):
    rows, cols = x.shape
    _ok(lib.rmsnorm_bwd(_ptr(dy, _BF, (rows, cols), "dy"), _ptr(x, _BF, name="x"),
                        _ptr(rstd, _F32, (rows,), "rstd"), _ptr(dx, _BF, (rows, cols), "dx"),
                        rows, cols, eps, _stream(stream)))


def mhc_layer_fwd(x, W, alpha3, b, f, bias, iters, eps_sk, eps_rms, H_pre, H_post, H_res,
                  u_save, r_save, y, out, ws, stream=None):
    T, n, C = x.shape
    O = _O(n)
    wp, wb = _ws(ws)
    _ok(lib.mhc_layer_fwd(
        _ptr(x, _BF, name="x"), _ptr(W, _F32, (n * C, O), "W"), _ptr(alpha3, _F32, (3,), "alpha3"),
        _ptr(b, _F32, (O,), "b"), _ptr(f, _BF, (T, C), "f"), _ptr(bias, _BF, (C,), "bias"),
        T, n, C, iters, eps_sk, eps_rms, _ptr(H_pre, _F32, (T, n), "H_pre"),
        _ptr(H_post, _F32, (T, n), "H_post"), _ptr(H_res, _F32, (T, n, n), "H_res"),
        _ptr(u_save, _F32, (T, O), "u_save"), _ptr(r_save, _F32, (T,), "r_save"),
        _ptr(y, _BF, (T, C), "y"), _ptr(out, _BF, (T, n, C), "out"), wp, wb, _stream(stream)))


def mhc_layer_bwd(dout, dy, x, W, alpha3, b, f, bias, H_pre, H_post, H_res, u_save, r_save,
                  iters, eps_sk, eps_rms, dx, df, dW, dalpha3, db, dbias, ws, stream=None):
    T, n, C = x.shape
    O = _O(n)
    wp, wb = _ws(ws)
    _ok(lib.mhc_layer_bwd(
        _ptr(dout, _BF, (T, n, C), "dout"), _ptr(dy, _BF, (T, C), "dy"), _ptr(x, _BF, name="x"),
        _ptr(W, _F32, (n * C, O), "W"), _ptr(alpha3, _F32, (3,), "alpha3"),
        _ptr(b, _F32, (O,), "b"), _ptr(f, _BF, (T, C), "f"), _ptr(bias, _BF, (C,), "bias"),
        _ptr(H_pre, _F32, (T, n), "H_pre"), _ptr(H_post, _F32, (T, n), "H_post"),
        _ptr(H_res, _F32, (T, n, n), "H_res"), _ptr(u_save, _F32, (T, O), "u_save"),
        _ptr(r_save, _F32, (T,), "r_save"), T, n, C, iters, eps_sk, eps_rms,
        _ptr(dx, _BF, (T, n, C), "dx"), _ptr(df, _BF, (T, C), "df"),
        _ptr(dW, _F32, (n * C, O), "dW"), _ptr(dalpha3, _F32, (3,), "dalpha3"),
        _ptr(db, _F32, (O,), "db"), _ptr(dbias, _F32, (C,), "dbias"), wp, wb, _stream(stream)))


def mhc_proj_rms_compute_h_fwd_noalloc(x, W, alpha3, b, iters, eps_sk, eps_rms, H_pre, H_post,
                                       H_res, u_save=None, r_save=None, stream=None):
    """mhc_proj_rms_compute_h_fwd with the library's fixed scratch array
    instead of a caller workspace (for callers that cannot allocate)."""
    T, n, C = x.shape
    O = _O(n)
    _ok(lib.mhc_proj_rms_compute_h_fwd_noalloc(
        _ptr(x, _BF, name="x"), _ptr(W, _F32, (n * C, O), "W"), _ptr(alpha3, _F32, (3,), "alpha3"),
        _ptr(b, _F32, (O,), "b"), T, n, C, iters, eps_sk, eps_rms,
        _ptr(H_pre, _F32, (T, n), "H_pre"), _ptr(H_post, _F32, (T, n), "H_post"),
        _ptr(H_res, _F32, (T, n, n), "H_res"), _ptr(u_save, _F32, (T, O), "u_save"),
        _ptr(r_save, _F32, (T,), "r_save"), _stream(stream)))


# ---------------------------------------------------------------------------
# ops beyond the layer path
# ---------------------------------------------------------------------------

def mhc_h_aggregate_static_fwd(x, H_pre, y, stream=None):
    T, n, C = x.shape
    _ok(lib.mhc_h_aggregate_static_fwd(_ptr(x, _BF, name="x"), _ptr(H_pre, _F32, (n,), "H_pre"),
                                       _ptr(y, _BF, (T, C), "y"), T, n, C, _stream(stream)))


def mhc_h_aggregate_static_bwd(dy, x, H_pre, dx, dH_pre, ws, stream=None):
    T, n, C = x.shape
    wp, wb = _ws(ws)
    _ok(lib.mhc_h_aggregate_static_bwd(
        _ptr(dy, _BF, (T, C), "dy"), _ptr(x, _BF, name="x"), _ptr(H_pre, _F32, (n,), "H_pre"),
        _ptr(dx, _BF, (T, n, C), "dx"), _ptr(dH_pre, _F32, (n,), "dH_pre"), T, n, C, wp, wb,
        _stream(stream)))


def rmsnorm_residual_fwd(x, res, gamma, h, y, rstd, eps, stream=None):
    rows, cols = x.shape
    _ok(lib.rmsnorm_residual_fwd(
        _ptr(x, _BF, name="x"), _ptr(res, _BF, (rows, cols), "res"),
        _ptr(gamma, _F32, (cols,), "gamma"), _ptr(h, _BF, (rows, cols), "h"),
        _ptr(y, _BF, (rows, cols), "y"), _ptr(rstd, _F32, (rows,), "rstd"), rows, cols, eps,
        _stream(stream)))


def rmsnorm_residual_bwd(dy, dh, x, res, gamma, rstd, dx, dgamma, eps, ws=None, stream=None):
    rows, cols = x.shape
    wp, wb = _ws(ws)
    _ok(lib.rmsnorm_residual_bwd(
        _ptr(dy, _BF, (rows, cols), "dy"), _ptr(dh, _BF, (rows, cols), "dh"),
        _ptr(x, _BF, name="x"), _ptr(res, _BF, (rows, cols), "res"),
        _ptr(gamma, _F32, (cols,), "gamma"), _ptr(rstd, _F32, (rows,), "rstd"),
        _ptr(dx, _BF, (rows, cols), "dx"), _ptr(dgamma, _F32, (cols,), "dgamma"), rows, cols,
        eps, wp, wb, _stream(stream)))


def mhc_h_aggregate_rmsnorm_fwd(x, H_pre, gamma, y, yn, rstd, eps, stream=None):
    T, n, C = x.shape
    _ok(lib.mhc_h_aggregate_rmsnorm_fwd(
        _ptr(x, _BF, name="x"), _ptr(H_pre, _F32, (T, n), "H_pre"),
        _ptr(gamma, _F32, (C,), "gamma"), _ptr(y, _BF, (T, C), "y"),
        _ptr(yn, _BF, (T, C), "yn"), _ptr(rstd, _F32, (T,), "rstd"), T, n, C, eps,
        _stream(stream)))


def mhc_h_aggregate_rmsnorm_bwd(dyn, dy, x, H_pre, gamma, rstd, dx, dH_pre, dgamma, eps,
                                ws=None, stream=None):
    T, n, C = x.shape
    wp, wb = _ws(ws)
    _ok(lib.mhc_h_aggregate_rmsnorm_bwd(
        _ptr(dyn, _BF, (T, C), "dyn"), _ptr(dy, _BF, (T, C), "dy"), _ptr(x, _BF, name="x"),
        _ptr(H_pre, _F32, (T, n), "H_pre"), _ptr(gamma, _F32, (C,), "gamma"),
        _ptr(rstd, _F32, (T,), "rstd"), _ptr(dx, _BF, (T, n, C), "dx"),
        _ptr(dH_pre, _F32, (T, n), "dH_pre"), _ptr(dgamma, _F32, (C,), "dgamma"), T, n, C, eps,
        wp, wb, _stream(stream)))


def mhc_proj_rms_partial_fwd(x_shard, W_shard, u_part, s_part, ws, stream=None):
    T, n, Cs = x_shard.shape
    O = _O(n)
    wp, wb = _ws(ws)
    _ok(lib.mhc_proj_rms_partial_fwd(
        _ptr(x_shard, _BF, name="x_shard"), _ptr(W_shard, _F32, (n * Cs, O), "W_shard"), T, n,
        Cs, _ptr(u_part, _F32, (T, O), "u_part"), _ptr(s_part, _F32, (T,), "s_part"), wp, wb,
        _stream(stream)))


def mhc_compute_h_fwd(u, s, K, alpha3, b, iters, eps_sk, eps_rms, H_pre, H_post, H_res, r_save,
                      stream=None):
    T, O = u.shape
    n = H_pre.shape[1]
    _ok(lib.mhc_compute_h_fwd(
        _ptr(u, _F32, (T, _O(n)), "u"), _ptr(s, _F32, (T,), "s"), K,
        _ptr(alpha3, _F32, (3,), "alpha3"), _ptr(b, _F32, (O,), "b"), T, n, iters, eps_sk,
        eps_rms, _ptr(H_pre, _F32, (T, n), "H_pre"), _ptr(H_post, _F32, (T, n), "H_post"),
        _ptr(H_res, _F32, (T, n, n), "H_res"), _ptr(r_save, _F32, (T,), "r_save"),
        _stream(stream)))


def mhc_compute_h_bwd(dH_pre, dH_post, dH_res, u, s, K, alpha3, b, iters, eps_sk, eps_rms, du,
                      coef, dalpha3, db, ws, stream=None):
    T, n = dH_pre.shape
    O = _O(n)
    wp, wb = _ws(ws)
    _ok(lib.mhc_compute_h_bwd(
        _ptr(dH_pre, _F32, (T, n), "dH_pre"), _ptr(dH_post, _F32, (T, n), "dH_post"),
        _ptr(dH_res, _F32, (T, n, n), "dH_res"), _ptr(u, _F32, (T, O), "u"),
        _ptr(s, _F32, (T,), "s"), K, _ptr(alpha3, _F32, (3,), "alpha3"),
        _ptr(b, _F32, (O,), "b"), T, n, iters, eps_sk, eps_rms, _ptr(du, _F32, (T, O), "du"),
        _ptr(coef, _F32, (T,), "coef"), _ptr(dalpha3, _F32, (3,), "dalpha3"),
        _ptr(db, _F32, (O,), "db"), wp, wb, _stream(stream)))


def mhc_proj_rms_partial_bwd(x_shard, W_shard, du, coef, dx_shard, dW_shard, ws, stream=None):
    T, n, Cs = x_shard.shape
    O = _O(n)
    wp, wb = _ws(ws)
    _ok(lib.mhc_proj_rms_partial_bwd(
        _ptr(x_shard, _BF, name="x_shard"), _ptr(W_shard, _F32, (n * Cs, O), "W_shard"),
        _ptr(du, _F32, (T, O), "du"), _ptr(coef, _F32, (T,), "coef"), T, n, Cs,
        _ptr(dx_shard, _BF, (T, n, Cs), "dx_shard"), _ptr(dW_shard, _F32, (n * Cs, O), "dW_shard"),
        wp, wb, _stream(stream)))


def mhc_set_batch_invariant(on: bool) -> None:
    lib.mhc_set_batch_invariant(1 if on else 0)


def mhc_batch_invariant() -> bool:
    return bool(lib.mhc_batch_invariant())


def mhc_set_pinned_reductions(on: bool) -> None:
    lib.mhc_set_pinned_reductions(1 if on else 0)


def mhc_pinned_reductions() -> bool:
    return bool(lib.mhc_pinned_reductions())
