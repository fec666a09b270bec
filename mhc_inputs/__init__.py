"""Seeded synthetic inputs for the mHC residual-stream ops.

This module holds no arithmetic of the method.  It draws random tensors with
the shapes and distributions of the workloads and hands the same bytes to both
the fp64 oracle and the CUDA library:

* generator: ``numpy.random.Generator(PCG64(seed))``;
* every draw is ``standard_normal`` in float32, then multiplied by its
  standard deviation;
* bf16 tensors are the round-to-nearest-even of those float32 values and are
  returned as ``uint16`` bit patterns (the exact bytes a bf16 tensor holds);
* draw order for a layer: x, f, bias, W, dout, dy, then (optional) b;
  a standalone RMSNorm pair (x_norm, dy_norm) is drawn after all of those.

Shapes follow the layer's notation: T tokens, n streams, C hidden size,
K = n*C, O = n*n + 2*n controller logits.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_bits",
    "bf16_bits_to_f32",
    "controller_width",
    "layer_inputs",
    "sinkhorn_inputs",
    "rmsnorm_inputs",
    "LAYER_WORKLOADS",
]


def controller_width(n: int) -> int:
    """Number of controller logits for n streams (pre n, post n, res n*n)."""
    return n * n + 2 * n


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return the bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact float32 value of bf16 bit patterns."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    a = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def layer_inputs(T: int, n: int, C: int, seed: int, *, w_std: float = 0.02,
                 alpha: float = 0.01, b_std: float = 0.0,
                 bias_std: float = 0.02, grads: bool = True,
                 rmsnorm: bool = False) -> dict:
    """Inputs of one mHC layer forward (+ backward upstream grads).

    Returns a dict with
      x     [T, n, C] bf16 bits  residual streams ~N(0,1)
      f     [T, C]    bf16 bits  sub-layer output ~N(0,1)
      bias  [C]       bf16 bits  ~N(0, bias_std)
      W     [K, O]    float32    controller projection ~N(0, w_std)
      alpha [3]       float32    (alpha_pre, alpha_post, alpha_res), all = alpha
      b     [O]       float32    controller bias: zeros, or ~N(0, b_std)
      dout  [T, n, C] bf16 bits  upstream grad of the post-mix output (grads)
      dy    [T, C]    bf16 bits  upstream grad of the aggregate output (grads)
      x_norm, dy_norm [T, C] bf16 bits  standalone RMSNorm pair (rmsnorm)
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    K, O = n * C, controller_width(n)
    out = {}
    out["x"] = bf16_bits(_normal(rng, (T, n, C), 1.0))
    out["f"] = bf16_bits(_normal(rng, (T, C), 1.0))
    out["bias"] = bf16_bits(_normal(rng, (C,), bias_std))
    out["W"] = _normal(rng, (K, O), w_std)
    if grads:
        out["dout"] = bf16_bits(_normal(rng, (T, n, C), 1.0))
        out["dy"] = bf16_bits(_normal(rng, (T, C), 1.0))
    out["alpha"] = np.full(3, alpha, dtype=np.float32)
    if b_std > 0.0:
        out["b"] = _normal(rng, (O,), b_std)
    else:
        out["b"] = np.zeros(O, dtype=np.float32)
    if rmsnorm:
        out["x_norm"] = bf16_bits(_normal(rng, (T, C), 1.0))
        out["dy_norm"] = bf16_bits(_normal(rng, (T, C), 1.0))
    return out


def sinkhorn_inputs(M: int, n: int, seed: int, *, std: float = 1.0) -> dict:
    """Batched Sinkhorn logits [M, n, n] ~N(0, std) and upstream grad ~N(0,1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return {
        "logits": _normal(rng, (M, n, n), std),
        "dP": _normal(rng, (M, n, n), 1.0),
    }


def rmsnorm_inputs(rows: int, cols: int, seed: int) -> dict:
    """Standalone RMSNorm input and upstream grad, both bf16 bits ~N(0,1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return {
        "x": bf16_bits(_normal(rng, (rows, cols), 1.0)),
        "dy": bf16_bits(_normal(rng, (rows, cols), 1.0)),
    }


def norm_inputs(rows: int, cols: int, seed: int, *, gamma_std: float = 0.1) -> dict:
    """rmsnorm_residual inputs: x, res, dy, dh bf16 bits ~N(0,1) and a
    per-channel weight gamma = 1 + N(0, gamma_std) in float32."""
    rng = np.random.Generator(np.random.PCG64(seed))
    out = {k: bf16_bits(_normal(rng, (rows, cols), 1.0)) for k in ("x", "res", "dy", "dh")}
    out["gamma"] = (np.float32(1.0) + _normal(rng, (cols,), gamma_std)).astype(np.float32)
    return out


def gate_inputs(T: int, n: int, seed: int) -> dict:
    """Aggregate weights in [0, 1): per-token H_pre [T, n] and one static
    H_pre [n], float32 uniform draws."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return {"H_pre": rng.random((T, n), dtype=np.float32),
            "H_static": rng.random(n, dtype=np.float32)}


def _load_spec() -> dict:
    import json
    import os
    path = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "configs",
                        "spec.json")
    with open(path) as fh:
        return json.load(fh)


# The fixed constants, readings, tolerances and workloads (configs/spec.json).
SPEC = _load_spec()
ITERS = int(SPEC["constants"]["sinkhorn_iters"])
EPS_SK = float(SPEC["constants"]["eps_sinkhorn"])
EPS_RMS = float(SPEC["constants"]["eps_rms"])
EPS_NORM = float(SPEC["constants"]["eps_rmsnorm"])

# The workloads, by what they are.  Each entry: (T, n, C, w_std, seed).
LAYER_WORKLOADS = {k: (v["T"], v["n"], v["C"], v["w_std"], v["seed"])
                   for k, v in SPEC["workloads"].items()}
