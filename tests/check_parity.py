"""Acceptance command: every boundary tensor of the hot path against the fp64
oracle, in the order the data flows, stopping at the first one that diverges.

    python tests/check_parity.py            # tiny shapes, n = 4 and n = 8
    python tests/check_parity.py --full     # plus the 7B-scale layer (sampled rows)

Prints one line per boundary (max error, allowed error) and exits 0 when all
pass; otherwise names the first diverging boundary and exits 1.  The
tolerances are those of configs/spec.json (the same rules as the GPU tests).
Needs a CUDA device and the built library; the oracle is compiled on demand.
"""
from __future__ import annotations

import argparse
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import mhc_inputs as mi  # noqa: E402

TOL = mi.SPEC["tolerances"]


def _err(kind, gpu, ref):
    g, r = np.asarray(gpu, dtype=np.float64), np.asarray(ref, dtype=np.float64)
    if not np.all(np.isfinite(g)):
        return float("inf"), 0.0
    e = float(np.max(np.abs(g - r))) if r.size else 0.0
    if kind == "H":
        return e, TOL["H_abs"]
    if kind == "bf16":  # |g - r| <= abs + rel |r|: report max(|g - r| - rel |r|) against abs
        return (float(np.max(np.abs(g - r) - TOL["bf16_rel"] * np.abs(r))) if r.size else 0.0,
                TOL["bf16_abs"])
    scale = float(np.max(np.abs(r))) if r.size else 0.0
    return e, TOL["fp32_rel_of_max"] * scale + TOL["fp32_abs"]


def boundaries(T, n, C, seed, sample=None):
    """(name, kind, gpu array, oracle array) in data-flow order."""
    import torch

    import layers_proj_rms_gb300 as M
    import oracle as orc
    from tests.test_gpu_ops import run_layer

    host = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    inp = mi.layer_inputs(T, n, C, seed)
    o = run_layer(M, inp, T, n, C)
    sub = inp
    idx = slice(None)
    if sample is not None:
        idx = sample
        sub = dict(inp)
        for k in ("x", "f", "dout", "dy"):
            sub[k] = inp[k][sample]
    f = orc.layer_fwd(sub, n, mi.ITERS, mi.EPS_SK, mi.EPS_RMS)
    b = orc.layer_bwd(sub, f, n, mi.ITERS, mi.EPS_SK, mi.EPS_RMS)
    tag = f"layer T={T} n={n} C={C}"
    ti = torch.from_numpy(np.asarray(idx)).cuda() if sample is not None else None
    pick = (lambda t: host(t[ti])) if sample is not None else host
    out = [(f"{tag}: fwd H_pre", "H", pick(o["H_pre"]), f["H_pre"]),
           (f"{tag}: fwd H_post", "H", pick(o["H_post"]), f["H_post"]),
           (f"{tag}: fwd H_res", "H", pick(o["H_res"]), f["H_res"]),
           (f"{tag}: fwd u", "fp32", pick(o["u"]), f["u"]),
           (f"{tag}: fwd y (aggregate)", "bf16", pick(o["y"]), f["y"]),
           (f"{tag}: fwd out (post_bda)", "bf16", pick(o["out"]), f["out"]),
           (f"{tag}: bwd df", "bf16", pick(o["df"]), b["df"]),
           (f"{tag}: bwd dx", "bf16", pick(o["dx"]), b["dx"])]
    if sample is None:
        out += [(f"{tag}: bwd dW", "fp32", host(o["dW"]), b["dW"]),
                (f"{tag}: bwd dalpha", "fp32", host(o["dalpha"]), b["dalpha"]),
                (f"{tag}: bwd db", "fp32", host(o["db"]), b["db"]),
                (f"{tag}: bwd dbias", "fp32", host(o["dbias"]), b["dbias"])]
    return out


def standalone(n):
    """Sinkhorn and RMSNorm boundaries."""
    import torch

    import layers_proj_rms_gb300 as M
    import oracle as orc
    host = lambda t: t.float().cpu().numpy().astype(np.float64)  # noqa: E731
    inp = mi.sinkhorn_inputs(333, n, 9)
    lg = torch.from_numpy(inp["logits"]).cuda()
    dP = torch.from_numpy(inp["dP"]).cuda()
    P, dl = torch.empty_like(lg), torch.empty_like(lg)
    M.mhc_sinkhorn_fwd(lg, P, mi.ITERS, mi.EPS_SK)
    M.mhc_sinkhorn_bwd(dP, lg, dl, mi.ITERS, mi.EPS_SK)
    rin = mi.norm_inputs(37, 264, 11)
    x = torch.from_numpy(rin["x"].view(np.int16)).view(torch.bfloat16).cuda()
    r = torch.from_numpy(rin["res"].view(np.int16)).view(torch.bfloat16).cuda()
    dy = torch.from_numpy(rin["dy"].view(np.int16)).view(torch.bfloat16).cuda()
    g = torch.from_numpy(rin["gamma"]).cuda()
    h, y, dx = torch.empty_like(x), torch.empty_like(x), torch.empty_like(x)
    rstd, dg = torch.empty(37, device="cuda"), torch.empty(264, device="cuda")
    M.rmsnorm_residual_fwd(x, r, g, h, y, rstd, mi.EPS_NORM)
    M.rmsnorm_residual_bwd(dy, None, x, r, g, rstd, dx, dg, mi.EPS_NORM,
                           M.workspace(M.OP_RMSNORM_RESIDUAL_BWD, 37, 0, 264))
    torch.cuda.synchronize()
    f64 = lambda bits: mi.bf16_bits_to_f32(bits).astype(np.float64)  # noqa: E731
    rf = orc.rmsnorm_residual_fwd(f64(rin["x"]), f64(rin["res"]), rin["gamma"].astype(np.float64),
                                  mi.EPS_NORM)
    rb = orc.rmsnorm_residual_bwd(f64(rin["dy"]), None, f64(rin["x"]), f64(rin["res"]),
                                  rin["gamma"].astype(np.float64), mi.EPS_NORM)
    return [(f"sinkhorn n={n}: fwd P", "H", host(P), orc.sinkhorn_fwd(inp["logits"], mi.ITERS, mi.EPS_SK)),
            (f"sinkhorn n={n}: bwd dlogits", "fp32", host(dl),
             orc.sinkhorn_bwd(inp["dP"], inp["logits"], mi.ITERS, mi.EPS_SK)),
            ("rmsnorm_residual: fwd h", "bf16", host(h), rf["h"]),
            ("rmsnorm_residual: fwd y", "bf16", host(y), rf["y"]),
            ("rmsnorm_residual: bwd dx", "bf16", host(dx), rb["dx"]),
            ("rmsnorm_residual: bwd dgamma", "fp32", host(dg), rb["dgamma"])]


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--full", action="store_true", help="also the 7B-scale layer, sampled rows")
    args = ap.parse_args()
    import torch
    if not torch.cuda.is_available():
        print("no CUDA device", file=sys.stderr)
        return 2
    checks = []
    checks += standalone(4) + standalone(8)
    checks += boundaries(256, 4, 256, 0)
    checks += boundaries(67, 8, 64, 4)
    if args.full:
        rows = np.unique(np.concatenate([[0, 16383], np.random.Generator(
            np.random.PCG64(1)).choice(16384, 32, replace=False)]))
        checks += boundaries(16384, 4, 4096, 3, sample=rows)
    for name, kind, gpu, ref in checks:
        err, allowed = _err(kind, gpu, ref)
        ok = err <= allowed
        print(f"{'ok  ' if ok else 'FAIL'} {name:44s} err {err:.3e}  allowed {allowed:.3e}")
        if not ok:
            print(f"first diverging boundary: {name}")
            return 1
    print(f"PASS: {len(checks)} boundaries")
    return 0


if __name__ == "__main__":
    sys.exit(main())
