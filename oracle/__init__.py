"""fp64 CPU oracle for the mHC residual-stream ops (test infrastructure).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg are the only code that may import this package.  The CUDA
library never calls it, and the two share no code; only the seeded input
generators in ``mhc_inputs`` feed both.

The arithmetic lives in ``mhc_oracle.c`` (plain C, double accumulators,
ascending loops, OpenMP over independent tokens).  This module compiles it
with gcc (``build()``) and wraps each entry point with numpy arrays.  The
layer composition (forward: proj_rms_compute_h, h_aggregate, h_post_bda;
backward: the three op backwards plus the three-way gradient sum) is written
out here from those functions.

Sources are the three web pages the C file names: the rwkv-ops mhu_ffi.cu
FFI handlers, the Megatron-Core ``core.fusions.fused_mhc_kernels`` API page,
and RL-Kernel PR #383 (P1 start kit for mHC + RMSNorm).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mhc_oracle.c")
_SRC_PINNED = os.path.join(_HERE, "mhc_oracle_pinned.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle_mhc.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no -ffast-math, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                    os.path.getmtime(_SRC_PINNED))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC",
           "-shared", "-Wall", "-o", tmp, _SRC, _SRC_PINNED, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _L():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        i64, i32, f64, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_double, ctypes.c_float
        P = ctypes.c_void_p
        sig = {
            "orc_sinkhorn_fwd": [P, P, i64, i32, i32, f64],
            "orc_sinkhorn_bwd": [P, P, P, i64, i32, i32, f64],
            "orc_proj_rms_compute_h_fwd": [P, P, P, P, i64, i32, i64, i32, f64, f64,
                                           P, P, P, P, P],
            "orc_proj_rms_compute_h_bwd": [P, P, P, P, P, P, P, i64, i32, i64, i32, f64,
                                           f64, P, P, P, P],
            "orc_h_aggregate_fwd": [P, P, i64, i32, i64, P],
            "orc_h_aggregate_bwd": [P, P, P, i64, i32, i64, P, P],
            "orc_h_post_bda_fwd": [P, P, P, P, P, i64, i32, i64, P],
            "orc_h_post_bda_bwd": [P, P, P, P, P, P, i64, i32, i64, P, P, P, P, P],
            "orc_rmsnorm_fwd": [P, i64, i64, f64, P, P],
            "orc_rmsnorm_bwd": [P, P, i64, i64, f64, P],
            "orc_h_aggregate_static_fwd": [P, P, i64, i32, i64, P],
            "orc_h_aggregate_static_bwd": [P, P, P, i64, i32, i64, P, P],
            "orc_rmsnorm_residual_fwd": [P, P, P, i64, i64, f64, P, P, P],
            "orc_rmsnorm_residual_bwd": [P, P, P, P, P, i64, i64, f64, P, P],
            "orc_proj_rms_partials": [P, P, i64, i32, i64, P, P],
            "orc_compute_h_from_sums": [P, P, i64, P, P, i64, i32, i32, f64, f64, P, P, P, P],
            "orc_compute_h_bwd_from_sums": [P, P, P, P, P, i64, P, P, i64, i32, i32, f64, f64,
                                            P, P, P, P],
            "orc_proj_rms_partial_bwd": [P, P, P, P, i64, i32, i64, P, P],
            "orc_num_threads": [],
            "orc_pin_sinkhorn_fwd": [P, P, i64, i32, f32],
            "orc_pin_sinkhorn_bwd": [P, P, P, i64, i32, f32, P],
            "orc_pin_proj_rms_compute_h_fwd": [P, P, P, P, i64, i64, i32, f32, f32, P, P, P, P, P],
            "orc_pin_proj_rms_compute_h_bwd": [P, P, P, P, P, P, P, i64, i64, i32, f32, f32,
                                               P, P, P, P, P, P],
            "orc_pin_h_aggregate_fwd": [P, P, i64, i64, P],
            "orc_pin_h_aggregate_bwd": [P, P, P, i64, i64, P, P],
            "orc_pin_h_post_bda_fwd": [P, P, P, P, P, i64, i64, P],
            "orc_pin_h_post_bda_bwd": [P, P, P, P, P, P, i64, i64, P, P, P, P, P],
            "orc_pin_layer_bwd": [P, P, P, P, P, P, P, P, P, P, P, i64, i64, i32, f32, f32, P, P,
                                  P, P, P, P, P, P],
        }
        for name, args in sig.items():
            fn = getattr(_lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        _lib.orc_pin_exp.argtypes = [f32]
        _lib.orc_pin_exp.restype = f32
    return _lib


def num_threads() -> int:
    """Threads the oracle's OpenMP regions use."""
    return int(_L().orc_num_threads())


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f64(a):
    """Any input as a contiguous float64 array.

    uint16 arrays are bf16 bit patterns and are widened exactly; float32 and
    float64 arrays are converted (exactly) as they are.
    """
    a = np.asarray(a)
    if a.dtype == np.uint16:
        a = (a.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return np.ascontiguousarray(a, dtype=np.float64)




def _check(rc, name):
    if rc != 0:
        raise RuntimeError(f"oracle {name} failed with code {rc}")


def controller_width(n):
    return n * n + 2 * n


# --------------------------------------------------------------------------
# Sinkhorn (rwkv-ops SinkhornFwdHost/BwdHost; Megatron fused_sinkhorn)
# --------------------------------------------------------------------------

def sinkhorn_fwd(logits, iters, eps):
    """P = Sinkhorn(exp(logits)) for logits [..., n, n]; returns fp64."""
    lg = _f64(logits)
    n = lg.shape[-1]
    M = lg.size // (n * n)
    P = np.empty(lg.shape, dtype=np.float64)
    _check(_L().orc_sinkhorn_fwd(_p(lg), _p(P), M, n, iters, float(eps)), "sinkhorn_fwd")
    return P


def sinkhorn_bwd(dP, logits, iters, eps):
    """Gradient of the unrolled Sinkhorn map with respect to the logits."""
    lg, g = _f64(logits), _f64(dP)
    n = lg.shape[-1]
    M = lg.size // (n * n)
    d = np.empty(lg.shape, dtype=np.float64)
    _check(_L().orc_sinkhorn_bwd(_p(g), _p(lg), _p(d), M, n, iters, float(eps)), "sinkhorn_bwd")
    return d


# --------------------------------------------------------------------------
# proj_rms_compute_h (Megatron fused_proj_rms_compute_h; RL-Kernel fp32_gemm_rms)
# --------------------------------------------------------------------------

def proj_rms_compute_h_fwd(x, W, alpha, b, n, iters, eps_sk, eps_rms):
    """x [T, n, C] (bf16 bits or float) -> dict(H_pre, H_post, H_res, u, r) in fp64."""
    x = _f64(x)
    T, C = x.shape[0], x.shape[-1]
    O = controller_width(n)
    H_pre = np.empty((T, n)); H_post = np.empty((T, n)); H_res = np.empty((T, n, n))
    u = np.empty((T, O)); r = np.empty(T)
    _check(_L().orc_proj_rms_compute_h_fwd(
        _p(x), _p(_f64(W)), _p(_f64(alpha)), _p(_f64(b)), T, n, C, iters, float(eps_sk),
        float(eps_rms), _p(H_pre), _p(H_post), _p(H_res), _p(u), _p(r)), "proj_fwd")
    return {"H_pre": H_pre, "H_post": H_post, "H_res": H_res, "u": u, "r": r}


def proj_rms_compute_h_bwd(dH_pre, dH_post, dH_res, x, W, alpha, b, n, iters, eps_sk,
                           eps_rms, *, want_dx=True, want_dW=True):
    """Returns dict(dx [T,n,C] or None, dW [K,O] or None, dalpha [3], db [O])."""
    x = _f64(x)
    T, C = x.shape[0], x.shape[-1]
    O = controller_width(n)
    dx = np.empty((T, n, C)) if want_dx else None
    dW = np.empty((n * C, O)) if want_dW else None
    dalpha = np.empty(3); db = np.empty(O)
    _check(_L().orc_proj_rms_compute_h_bwd(
        _p(_f64(dH_pre)), _p(_f64(dH_post)), _p(_f64(dH_res)), _p(x), _p(_f64(W)),
        _p(_f64(alpha)), _p(_f64(b)), T, n, C, iters, float(eps_sk), float(eps_rms),
        _p(dx), _p(dW), _p(dalpha), _p(db)), "proj_bwd")
    return {"dx": dx, "dW": dW, "dalpha": dalpha, "db": db}


# --------------------------------------------------------------------------
# h_aggregate (Megatron fused_h_aggregate / FusedHAggregate; rwkv StreamAggregate)
# --------------------------------------------------------------------------

def h_aggregate_fwd(x, H_pre):
    x = _f64(x)
    T, n, C = x.shape
    y = np.empty((T, C))
    _check(_L().orc_h_aggregate_fwd(_p(x), _p(_f64(H_pre)), T, n, C, _p(y)), "agg_fwd")
    return y


def h_aggregate_bwd(dy, x, H_pre, *, want_dx=True):
    x = _f64(x)
    T, n, C = x.shape
    dx = np.empty((T, n, C)) if want_dx else None
    dH = np.empty((T, n))
    _check(_L().orc_h_aggregate_bwd(_p(_f64(dy)), _p(x), _p(_f64(H_pre)), T, n, C, _p(dx),
                                    _p(dH)), "agg_bwd")
    return {"dx": dx, "dH_pre": dH}


# --------------------------------------------------------------------------
# h_post_bda (Megatron fused_h_post_bda / _torch_h_post_bda_bwd; rwkv MhcPostOp)
# --------------------------------------------------------------------------

def h_post_bda_fwd(res, f, bias, H_res, H_post):
    res = _f64(res)
    T, n, C = res.shape
    out = np.empty((T, n, C))
    _check(_L().orc_h_post_bda_fwd(_p(res), _p(_f64(f)), _p(None if bias is None else _f64(bias)),
                                   _p(_f64(H_res)), _p(_f64(H_post)), T, n, C, _p(out)),
           "post_fwd")
    return out


def h_post_bda_bwd(dout, res, f, bias, H_res, H_post, *, want_dres=True, want_df=True,
                   want_dbias=True):
    res = _f64(res)
    T, n, C = res.shape
    dres = np.empty((T, n, C)) if want_dres else None
    df = np.empty((T, C)) if want_df else None
    dbias = np.empty(C) if want_dbias else None
    dHres = np.empty((T, n, n)); dHpost = np.empty((T, n))
    _check(_L().orc_h_post_bda_bwd(
        _p(_f64(dout)), _p(res), _p(_f64(f)), _p(None if bias is None else _f64(bias)),
        _p(_f64(H_res)), _p(_f64(H_post)), T, n, C, _p(dres), _p(df), _p(dbias), _p(dHres),
        _p(dHpost)), "post_bwd")
    return {"dres": dres, "df": df, "dbias": dbias, "dH_res": dHres, "dH_post": dHpost}


# --------------------------------------------------------------------------
# Standalone RMSNorm (rwkv RMSNormFwdHost / RMSNormBwdHost)
# --------------------------------------------------------------------------

def rmsnorm_fwd(x, eps):
    x = _f64(x)
    rows, cols = x.shape
    y = np.empty((rows, cols)); rstd = np.empty(rows)
    _check(_L().orc_rmsnorm_fwd(_p(x), rows, cols, float(eps), _p(y), _p(rstd)), "rms_fwd")
    return y, rstd


def rmsnorm_bwd(dy, x, eps):
    x = _f64(x)
    rows, cols = x.shape
    dx = np.empty((rows, cols))
    _check(_L().orc_rmsnorm_bwd(_p(_f64(dy)), _p(x), rows, cols, float(eps), _p(dx)), "rms_bwd")
    return dx


# --------------------------------------------------------------------------
# h_aggregate with a static (token-independent) H_pre [n] (rwkv
# StreamAggregateFwd/Bwd with per_token = false)
# --------------------------------------------------------------------------

def h_aggregate_static_fwd(x, H_pre):
    x = _f64(x)
    T, n, C = x.shape
    y = np.empty((T, C))
    _check(_L().orc_h_aggregate_static_fwd(_p(x), _p(_f64(H_pre)), T, n, C, _p(y)), "aggs_fwd")
    return y


def h_aggregate_static_bwd(dy, x, H_pre, *, want_dx=True):
    x = _f64(x)
    T, n, C = x.shape
    dx = np.empty((T, n, C)) if want_dx else None
    dH = np.empty(n)
    _check(_L().orc_h_aggregate_static_bwd(_p(_f64(dy)), _p(x), _p(_f64(H_pre)), T, n, C,
                                           _p(dx), _p(dH)), "aggs_bwd")
    return {"dx": dx, "dH_pre": dH}


# --------------------------------------------------------------------------
# rmsnorm_residual (RL-Kernel PR #383 task P1-5 "RMSNorm + residual fork",
# P1-8 "cross-rank dgamma"): h = x + res, y = h rho gamma
# --------------------------------------------------------------------------

def rmsnorm_residual_fwd(x, res, gamma, eps):
    x = _f64(x)
    rows, cols = x.shape
    h = np.empty((rows, cols)); y = np.empty((rows, cols)); rstd = np.empty(rows)
    _check(_L().orc_rmsnorm_residual_fwd(_p(x), _p(None if res is None else _f64(res)),
                                         _p(None if gamma is None else _f64(gamma)), rows, cols,
                                         float(eps), _p(h), _p(y), _p(rstd)), "rmsr_fwd")
    return {"h": h, "y": y, "rstd": rstd}


def rmsnorm_residual_bwd(dy, dh, x, res, gamma, eps):
    x = _f64(x)
    rows, cols = x.shape
    dx = np.empty((rows, cols)); dgamma = np.empty(cols)
    _check(_L().orc_rmsnorm_residual_bwd(_p(_f64(dy)), _p(None if dh is None else _f64(dh)),
                                         _p(x), _p(None if res is None else _f64(res)),
                                         _p(None if gamma is None else _f64(gamma)), rows, cols,
                                         float(eps), _p(dx), _p(dgamma)), "rmsr_bwd")
    return {"dx": dx, "dgamma": dgamma}


# --------------------------------------------------------------------------
# h_aggregate followed by the weighted RMSNorm of its output, as one op:
# y = sum_i H_pre[i] x_i (kept: the pre-normalization intermediate) and
# yn = y rho gamma.  Backward: the gradient at y is dy (if y is used
# elsewhere) plus the RMSNorm backward of dyn; then the aggregate backward.
# --------------------------------------------------------------------------

def h_aggregate_rmsnorm_fwd(x, H_pre, gamma, eps):
    y = h_aggregate_fwd(x, H_pre)
    r = rmsnorm_residual_fwd(y, None, gamma, eps)
    return {"y": y, "yn": r["y"], "rstd": r["rstd"]}


def h_aggregate_rmsnorm_bwd(dyn, dy, x, H_pre, gamma, eps):
    y = h_aggregate_fwd(x, H_pre)
    r = rmsnorm_residual_bwd(dyn, dy, y, None, gamma, eps)
    a = h_aggregate_bwd(r["dx"], x, H_pre)
    return {"dx": a["dx"], "dH_pre": a["dH_pre"], "dgamma": r["dgamma"]}


# --------------------------------------------------------------------------
# proj_rms_compute_h over channel shards (RL-Kernel PR #383 task P1-6, the
# fp32_gemm_rms TP/SP contract): per-shard partial sums, compute_h on the
# totals, per-shard backward from the per-token du and RMS coefficient.
# --------------------------------------------------------------------------

def proj_rms_partials(xs, Ws):
    xs = _f64(xs)
    T, n, Cs = xs.shape
    O = controller_width(n)
    u = np.empty((T, O)); s = np.empty(T)
    _check(_L().orc_proj_rms_partials(_p(xs), _p(_f64(Ws)), T, n, Cs, _p(u), _p(s)), "partials")
    return {"u": u, "s": s}


def compute_h_from_sums(u, s, K, alpha, b, n, iters, eps_sk, eps_rms):
    u = _f64(u)
    T = u.shape[0]
    H_pre = np.empty((T, n)); H_post = np.empty((T, n)); H_res = np.empty((T, n, n))
    r = np.empty(T)
    _check(_L().orc_compute_h_from_sums(_p(u), _p(_f64(s)), K, _p(_f64(alpha)), _p(_f64(b)), T,
                                        n, iters, eps_sk, eps_rms, _p(H_pre), _p(H_post),
                                        _p(H_res), _p(r)), "compute_h_sums")
    return {"H_pre": H_pre, "H_post": H_post, "H_res": H_res, "r": r}


def compute_h_bwd_from_sums(dH_pre, dH_post, dH_res, u, s, K, alpha, b, n, iters, eps_sk,
                            eps_rms):
    u = _f64(u)
    T, O = u.shape
    du = np.empty((T, O)); coef = np.empty(T); dalpha = np.empty(3); db = np.empty(O)
    _check(_L().orc_compute_h_bwd_from_sums(_p(_f64(dH_pre)), _p(_f64(dH_post)),
                                            _p(_f64(dH_res)), _p(u), _p(_f64(s)), K,
                                            _p(_f64(alpha)), _p(_f64(b)), T, n, iters, eps_sk,
                                            eps_rms, _p(du), _p(coef), _p(dalpha), _p(db)),
           "compute_h_bwd_sums")
    return {"du": du, "coef": coef, "dalpha": dalpha, "db": db}


def proj_rms_partial_bwd(xs, Ws, du, coef):
    xs = _f64(xs)
    T, n, Cs = xs.shape
    O = controller_width(n)
    dx = np.empty((T, n, Cs)); dW = np.empty((n * Cs, O))
    _check(_L().orc_proj_rms_partial_bwd(_p(xs), _p(_f64(Ws)), _p(_f64(du)), _p(_f64(coef)), T,
                                         n, Cs, _p(dx), _p(dW)), "partial_bwd")
    return {"dx": dx, "dW": dW}


# --------------------------------------------------------------------------
# One mHC layer: forward = proj_rms_compute_h -> h_aggregate -> h_post_bda
# (Megatron fused_mhc_kernels: the four fused ops); backward = the three op
# backwards and the three-way sum of the residual gradient (fused_add_3).
# f (the sub-layer output) and the upstream grads dout, dy are inputs.
# --------------------------------------------------------------------------

def layer_fwd(inp, n, iters, eps_sk, eps_rms):
    h = proj_rms_compute_h_fwd(inp["x"], inp["W"], inp["alpha"], inp["b"], n, iters, eps_sk,
                               eps_rms)
    y = h_aggregate_fwd(inp["x"], h["H_pre"])
    out = h_post_bda_fwd(inp["x"], inp["f"], inp["bias"], h["H_res"], h["H_post"])
    return dict(h, y=y, out=out)


def layer_bwd(inp, fwd, n, iters, eps_sk, eps_rms, *, want_dx=True):
    """Gradients of L = <dout, out> + <dy, y> for one layer.

    With want_dx=False only the per-token reductions and the parameter grads
    are formed (dW, dalpha, db, dbias); the [T, n, C] and [T, C] tensors are
    skipped, which lets full-size runs stay within host memory.
    """
    pb = h_post_bda_bwd(inp["dout"], inp["x"], inp["f"], inp["bias"], fwd["H_res"],
                        fwd["H_post"], want_dres=want_dx, want_df=want_dx)
    ab = h_aggregate_bwd(inp["dy"], inp["x"], fwd["H_pre"], want_dx=want_dx)
    prb = proj_rms_compute_h_bwd(ab["dH_pre"], pb["dH_post"], pb["dH_res"], inp["x"], inp["W"],
                                 inp["alpha"], inp["b"], n, iters, eps_sk, eps_rms,
                                 want_dx=want_dx)
    res = {"dW": prb["dW"], "dalpha": prb["dalpha"], "db": prb["db"], "dbias": pb["dbias"],
           "dH_pre": ab["dH_pre"], "dH_post": pb["dH_post"], "dH_res": pb["dH_res"]}
    if want_dx:
        res["dx"] = pb["dres"] + ab["dx"] + prb["dx"]
        res["df"] = pb["df"]
    return res


# --------------------------------------------------------------------------
# Cross-layer fusion (RL-Kernel PR #383 body: fuse fp32_gemm_rms with the op
# that produces its input): the post-mix of layer l feeds layer l+1's
# proj_rms_compute_h.  Layer l+1 reads layer l's output as it is stored, i.e.
# after the single bf16 round-to-nearest-even of the post-mix (the only
# rounding of a bf16 output); its H follows from that input.
# --------------------------------------------------------------------------

def bf16_rne(a):
    """Round fp64 values to the nearest bf16 value, ties to even (8
    significant bits; exponent range of fp32, subnormal spacing 2^-133);
    returned as fp64.  Written from the definition: with e = floor(log2|v|)
    (at least -126), the bf16 values near v are the multiples of 2^(e-7)."""
    v = np.asarray(a, dtype=np.float64)
    out = np.zeros_like(v)
    nz = v != 0
    e = np.floor(np.log2(np.abs(v[nz])))
    # log2 may land one off next to a power of two; fix e so 2^e <= |v| < 2^(e+1)
    e = np.where(np.abs(v[nz]) < np.exp2(e), e - 1, e)
    e = np.where(np.abs(v[nz]) >= np.exp2(e + 1), e + 1, e)
    e = np.maximum(e, -126.0)
    ulp = np.exp2(e - 7)
    out[nz] = np.rint(v[nz] / ulp) * ulp  # np.rint: round half to even
    return out


def h_post_bda_compute_h_fwd(res, f, bias, H_res, H_post, W_next, alpha_next, b_next, n, iters,
                             eps_sk, eps_rms):
    out = h_post_bda_fwd(res, f, bias, H_res, H_post)
    x_next = bf16_rne(out)
    h = proj_rms_compute_h_fwd(x_next, W_next, alpha_next, b_next, n, iters, eps_sk, eps_rms)
    return dict(h, out=out, x_next=x_next)


# --------------------------------------------------------------------------
# fp32, pinned reduction order (mhc_oracle_pinned.c): the reference of the
# library's bit-reproducible mode, n = 4.  RL-Kernel PR #383, PR body,
# "Numerical contract": a serial ascending left fold for long reductions,
# (a0 + a1) + (a2 + a3) over the four streams, fp32 arithmetic.
# Inputs are the exact fp32 values (bf16 bit patterns are widened); bf16
# outputs come back as their fp32 values.
# --------------------------------------------------------------------------

def _f32(a):
    a = np.asarray(a)
    if a.dtype == np.uint16:
        a = (a.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return np.ascontiguousarray(a, dtype=np.float32)


def pin_exp(x):
    """The exp of the pinned mode (Cody-Waite reduction, Taylor degree 7), elementwise."""
    L = _L()
    return np.array([L.orc_pin_exp(float(v)) for v in np.asarray(x, dtype=np.float32).ravel()],
                    dtype=np.float32).reshape(np.shape(x))


def pin_sinkhorn_fwd(logits, iters, eps):
    lg = _f32(logits)
    M = lg.size // 16
    P = np.empty_like(lg)
    _check(_L().orc_pin_sinkhorn_fwd(_p(lg), _p(P), M, iters, eps), "pin_sinkhorn_fwd")
    return P


def pin_sinkhorn_bwd(dP, logits, iters, eps):
    lg, g = _f32(logits), _f32(dP)
    M = lg.size // 16
    dl = np.empty_like(lg)
    trace = np.empty((2 * iters + 1) * 16, dtype=np.float32)
    _check(_L().orc_pin_sinkhorn_bwd(_p(g), _p(lg), _p(dl), M, iters, eps, _p(trace)),
           "pin_sinkhorn_bwd")
    return dl


def pin_proj_rms_compute_h_fwd(x, W, alpha, b, iters, eps_sk, eps_rms):
    xs, Ws, a, bb = _f32(x), _f32(W), _f32(alpha), _f32(b)
    T, n, C = xs.shape
    assert n == 4
    out = {"H_pre": np.empty((T, 4), np.float32), "H_post": np.empty((T, 4), np.float32),
           "H_res": np.empty((T, 4, 4), np.float32), "u": np.empty((T, 24), np.float32),
           "r": np.empty(T, np.float32)}
    _check(_L().orc_pin_proj_rms_compute_h_fwd(
        _p(xs), _p(Ws), _p(a), _p(bb), T, C, iters, eps_sk, eps_rms, _p(out["H_pre"]),
        _p(out["H_post"]), _p(out["H_res"]), _p(out["u"]), _p(out["r"])), "pin_proj_fwd")
    return out


def pin_proj_rms_compute_h_bwd(dHpre, dHpost, dHres, x, W, alpha, b, iters, eps_sk, eps_rms):
    xs, Ws, a, bb = _f32(x), _f32(W), _f32(alpha), _f32(b)
    T, n, C = xs.shape
    out = {"dx": np.empty((T, 4, C), np.float32), "dW": np.empty((4 * C, 24), np.float32),
           "dalpha": np.empty(3, np.float32), "db": np.empty(24, np.float32)}
    scratch = np.empty(max(T, 1) * (2 * 24 + 4), np.float32)
    trace = np.empty((2 * iters + 1) * 16, np.float32)
    _check(_L().orc_pin_proj_rms_compute_h_bwd(
        _p(_f32(dHpre)), _p(_f32(dHpost)), _p(_f32(dHres)), _p(xs), _p(Ws), _p(a), _p(bb), T, C,
        iters, eps_sk, eps_rms, _p(out["dx"]), _p(out["dW"]), _p(out["dalpha"]), _p(out["db"]),
        _p(scratch), _p(trace)), "pin_proj_bwd")
    return out


def pin_h_aggregate_fwd(x, H_pre):
    xs = _f32(x)
    T, n, C = xs.shape
    y = np.empty((T, C), np.float32)
    _check(_L().orc_pin_h_aggregate_fwd(_p(xs), _p(_f32(H_pre)), T, C, _p(y)), "pin_agg_fwd")
    return y


def pin_h_aggregate_bwd(dy, x, H_pre):
    xs = _f32(x)
    T, n, C = xs.shape
    dx = np.empty((T, 4, C), np.float32)
    dH = np.empty((T, 4), np.float32)
    _check(_L().orc_pin_h_aggregate_bwd(_p(_f32(dy)), _p(xs), _p(_f32(H_pre)), T, C, _p(dx),
                                        _p(dH)), "pin_agg_bwd")
    return dx, dH


def pin_h_post_bda_fwd(res, f, bias, H_res, H_post):
    rs = _f32(res)
    T, n, C = rs.shape
    out = np.empty((T, 4, C), np.float32)
    _check(_L().orc_pin_h_post_bda_fwd(_p(rs), _p(_f32(f)), _p(None if bias is None else _f32(bias)),
                                       _p(_f32(H_res)), _p(_f32(H_post)), T, C, _p(out)),
           "pin_post_fwd")
    return out


def pin_h_post_bda_bwd(dout, res, f, bias, H_res, H_post):
    rs = _f32(res)
    T, n, C = rs.shape
    o = {"dres": np.empty((T, 4, C), np.float32), "df": np.empty((T, C), np.float32),
         "dbias": np.empty(C, np.float32), "dH_res": np.empty((T, 4, 4), np.float32),
         "dH_post": np.empty((T, 4), np.float32)}
    _check(_L().orc_pin_h_post_bda_bwd(
        _p(_f32(dout)), _p(rs), _p(_f32(f)), _p(None if bias is None else _f32(bias)),
        _p(_f32(H_res)), _p(_f32(H_post)), T, C, _p(o["dres"]), _p(o["df"]), _p(o["dbias"]),
        _p(o["dH_res"]), _p(o["dH_post"])), "pin_post_bwd")
    return o


def pin_layer_fwd(inp, iters, eps_sk, eps_rms):
    """The layer forward in the pinned order: proj_rms_compute_h, then
    h_aggregate and h_post_bda with its H."""
    h = pin_proj_rms_compute_h_fwd(inp["x"], inp["W"], inp["alpha"], inp["b"], iters, eps_sk,
                                   eps_rms)
    h["y"] = pin_h_aggregate_fwd(inp["x"], h["H_pre"])
    h["out"] = pin_h_post_bda_fwd(inp["x"], inp["f"], inp.get("bias"), h["H_res"], h["H_post"])
    return h


def pin_layer_bwd(inp, fwd, iters, eps_sk, eps_rms):
    xs = _f32(inp["x"])
    T, n, C = xs.shape
    o = {"dx": np.empty((T, 4, C), np.float32), "df": np.empty((T, C), np.float32),
         "dW": np.empty((4 * C, 24), np.float32), "dalpha": np.empty(3, np.float32),
         "db": np.empty(24, np.float32), "dbias": np.empty(C, np.float32)}
    scratch = np.empty(max(T, 1) * (2 * 24 + 4 + 8 + 16), np.float32)
    trace = np.empty((2 * iters + 1) * 16, np.float32)
    bias = inp.get("bias")
    _check(_L().orc_pin_layer_bwd(
        _p(_f32(inp["dout"])), _p(_f32(inp["dy"])), _p(xs), _p(_f32(inp["W"])),
        _p(_f32(inp["alpha"])), _p(_f32(inp["b"])), _p(_f32(inp["f"])),
        _p(None if bias is None else _f32(bias)), _p(_f32(fwd["H_pre"])), _p(_f32(fwd["H_post"])),
        _p(_f32(fwd["H_res"])), T, C, iters, eps_sk, eps_rms, _p(o["dx"]), _p(o["df"]),
        _p(o["dW"]), _p(o["dalpha"]), _p(o["db"]), _p(o["dbias"]), _p(scratch), _p(trace)),
        "pin_layer_bwd")
    return o
