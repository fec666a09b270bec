"""Helpers shared by the tests: device transfer of seeded inputs and the
tolerance rules of the parity checks.

Tolerances (GPU result vs the fp64 oracle):
  * fp32 H tensors (H_pre, H_post, H_res, Sinkhorn P): |err| <= 1e-5.
  * bf16 activations and gradients: |err| <= 2e-2 + 1e-2 |ref|.
  * fp32 gradient tensors and other fp32 outputs: |err| <= 1e-4 max|ref| + 1e-5
    (a sum of C products of size ~1 carries fp32 rounding far above 1e-5).
"""
from __future__ import annotations

import numpy as np
import torch

import mhc_inputs as mi

_TOL = mi.SPEC["tolerances"]


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """bf16 bit patterns (uint16) -> CUDA bf16 tensor with the same bytes."""
    a = np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(a).view(torch.bfloat16).cuda()


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def err_h(gpu, ref, tol=_TOL["H_abs"]):
    g, r = host(gpu) if isinstance(gpu, torch.Tensor) else gpu, np.asarray(ref)
    err = float(np.max(np.abs(g - r))) if r.size else 0.0
    assert np.all(np.isfinite(g)), "non-finite values"
    assert err <= tol, f"fp32 H mismatch: max abs err {err:.3e} > {tol:.1e}"
    return err


def err_bf16(gpu, ref, atol=_TOL["bf16_abs"], rtol=_TOL["bf16_rel"]):
    g, r = host(gpu) if isinstance(gpu, torch.Tensor) else gpu, np.asarray(ref)
    assert np.all(np.isfinite(g)), "non-finite values"
    if not r.size:
        return 0.0
    excess = np.abs(g - r) - (atol + rtol * np.abs(r))
    worst = float(np.max(excess))
    assert worst <= 0.0, (f"bf16 mismatch: max excess {worst:.3e} at "
                          f"{np.unravel_index(np.argmax(excess), r.shape)}")
    return float(np.max(np.abs(g - r)))


def err_grad(gpu, ref, rel=_TOL["fp32_rel_of_max"], atol=_TOL["fp32_abs"]):
    g, r = host(gpu) if isinstance(gpu, torch.Tensor) else gpu, np.asarray(ref)
    assert np.all(np.isfinite(g)), "non-finite values"
    if not r.size:
        return 0.0
    scale = float(np.max(np.abs(r)))
    err = float(np.max(np.abs(g - r)))
    assert err <= rel * scale + atol, f"fp32 grad mismatch: err {err:.3e}, max|ref| {scale:.3e}"
    return err
