"""GPU parity of the ops beyond the layer path against the fp64 oracle, on
the same seeded inputs, with out-of-bounds canaries around the outputs:

  * h_aggregate with a static H_pre [n] (rwkv-ops StreamAggregate with
    per_token = false);
  * rmsnorm_residual (RL-Kernel PR #383 tasks P1-5 / P1-8: residual fork,
    learnable gamma, dgamma);
  * h_aggregate fused with the weighted RMSNorm of its output;
  * proj_rms_compute_h over channel shards (task P1-6): shard partial sums,
    compute_h on the summed totals, per-token backward coefficients, a
    shard's dx and dW; the shards assembled against the unsharded oracle.

Sizes span several blocks with ragged tails; the full 7B-scale sizes are
checked on sampled rows where the oracle would be slow.
"""
import numpy as np
import pytest
import torch

import mhc_inputs as mi
from tests._util import dev_bf16, dev_f32, err_bf16, err_grad, err_h, host
from tests.test_gpu_ops import EPS_RMS, EPS_SK, ITERS, canary, check_canary

pytestmark = pytest.mark.gpu
EPS_N = 1e-6


@pytest.fixture(scope="module")
def M():
    import layers_proj_rms_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return m


def _f64(bits):
    return mi.bf16_bits_to_f32(bits).astype(np.float64)


# ---------------------------------------------------------------------------
# static H_pre
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,n,C", [(1, 4, 8), (129, 4, 264), (67, 8, 64), (300, 8, 136),
                                   (2048, 4, 4096)])
def test_aggregate_static(M, orc, T, n, C):
    inp = mi.layer_inputs(T, n, C, 200 + T, grads=True)
    H = mi.gate_inputs(T, n, 201 + T)["H_static"]
    x, dy = dev_bf16(inp["x"]), dev_bf16(inp["dy"])
    Hd = dev_f32(H)
    by, y = canary((T, C), torch.bfloat16)
    bx, dx = canary((T, n, C), torch.bfloat16)
    bh, dH = canary((n,), torch.float32)
    ws = M.workspace(M.OP_H_AGGREGATE_STATIC_BWD, T, n, C)
    M.mhc_h_aggregate_static_fwd(x, Hd, y)
    M.mhc_h_aggregate_static_bwd(dy, x, Hd, dx, dH, ws)
    torch.cuda.synchronize()
    for b in (by, bx, bh):
        check_canary(b)
    xf = _f64(inp["x"])
    err_bf16(y, orc.h_aggregate_static_fwd(xf, H))
    ref = orc.h_aggregate_static_bwd(_f64(inp["dy"]), xf, H)
    err_bf16(dx, ref["dx"])
    err_grad(dH, ref["dH_pre"])


def test_aggregate_static_zero_tokens(M):
    dH = torch.full((4,), 5.0, device="cuda")
    e = torch.empty(0, dtype=torch.bfloat16, device="cuda")
    M.mhc_h_aggregate_static_bwd(e.view(0, 64), e.view(0, 4, 64), torch.ones(4, device="cuda"),
                                 e.view(0, 4, 64), dH, None)
    torch.cuda.synchronize()
    assert torch.all(dH == 0)


# ---------------------------------------------------------------------------
# rmsnorm_residual
# ---------------------------------------------------------------------------

NORM_SHAPES = [(1, 8), (3, 264), (200, 1024), (67, 4096), (33, 7168), (5, 32768)]


@pytest.mark.parametrize("rows,cols", NORM_SHAPES)
@pytest.mark.parametrize("variant", ["res_gamma", "plain", "gamma_no_rstd"])
def test_rmsnorm_residual(M, orc, rows, cols, variant):
    inp = mi.norm_inputs(rows, cols, 300 + rows + cols)
    with_res = variant == "res_gamma"
    with_gamma = variant != "plain"
    x, dy, dh = dev_bf16(inp["x"]), dev_bf16(inp["dy"]), dev_bf16(inp["dh"])
    res = dev_bf16(inp["res"]) if with_res else None
    gamma = dev_f32(inp["gamma"]) if with_gamma else None
    bh, h = canary((rows, cols), torch.bfloat16)
    byy, y = canary((rows, cols), torch.bfloat16)
    br, rstd = canary((rows,), torch.float32)
    bdx, dx = canary((rows, cols), torch.bfloat16)
    bg, dg = canary((cols,), torch.float32)
    M.rmsnorm_residual_fwd(x, res, gamma, h, y, rstd, EPS_N)
    ws = M.workspace(M.OP_RMSNORM_RESIDUAL_BWD, rows, 0, cols)
    M.rmsnorm_residual_bwd(dy, dh if with_res else None, x, res, gamma,
                           None if variant == "gamma_no_rstd" else rstd, dx, dg, EPS_N, ws)
    torch.cuda.synchronize()
    for b in (bh, byy, br, bdx, bg):
        check_canary(b)
    xf = _f64(inp["x"]); rf = _f64(inp["res"]) if with_res else None
    gf = inp["gamma"].astype(np.float64) if with_gamma else None
    f = orc.rmsnorm_residual_fwd(xf, rf, gf, EPS_N)
    err_bf16(h, f["h"])
    err_bf16(y, f["y"])
    err_grad(rstd, f["rstd"], rel=1e-5)
    b = orc.rmsnorm_residual_bwd(_f64(inp["dy"]), _f64(inp["dh"]) if with_res else None, xf, rf,
                                 gf, EPS_N)
    err_bf16(dx, b["dx"])
    err_grad(dg, b["dgamma"])


def test_rmsnorm_residual_zero_row(M, orc):
    """An all-zero fork row: finite, y = 0, dx = rho g (rho = 1/sqrt(eps))."""
    inp = mi.norm_inputs(4, 64, 7)
    xb = inp["x"].copy(); xb[1] = 0
    rb = np.zeros_like(inp["res"])
    x, res = dev_bf16(xb), dev_bf16(rb)
    gamma, dy = dev_f32(inp["gamma"]), dev_bf16(inp["dy"])
    h = torch.empty(4, 64, dtype=torch.bfloat16, device="cuda")
    y, dx = torch.empty_like(h), torch.empty_like(h)
    rstd = torch.empty(4, device="cuda"); dg = torch.empty(64, device="cuda")
    M.rmsnorm_residual_fwd(x, res, gamma, h, y, rstd, EPS_N)
    M.rmsnorm_residual_bwd(dy, None, x, res, gamma, rstd, dx, dg, EPS_N,
                           M.workspace(M.OP_RMSNORM_RESIDUAL_BWD, 4, 0, 64))
    torch.cuda.synchronize()
    f = orc.rmsnorm_residual_fwd(_f64(xb), _f64(rb), inp["gamma"].astype(np.float64), EPS_N)
    b = orc.rmsnorm_residual_bwd(_f64(inp["dy"]), None, _f64(xb), _f64(rb),
                                 inp["gamma"].astype(np.float64), EPS_N)
    assert torch.all(torch.isfinite(dx.float()))
    err_bf16(y, f["y"])
    err_bf16(dx, b["dx"])  # rho = 1/sqrt(eps): the zero row has |dx| ~ 1e3
    err_grad(dg, b["dgamma"])


def test_rmsnorm_residual_7b_rows_sampled(M, orc):
    rows, cols = 16384, 4096
    inp = mi.norm_inputs(rows, cols, 77)
    x, res, dy = dev_bf16(inp["x"]), dev_bf16(inp["res"]), dev_bf16(inp["dy"])
    gamma = dev_f32(inp["gamma"])
    h = torch.empty(rows, cols, dtype=torch.bfloat16, device="cuda")
    y, dx = torch.empty_like(h), torch.empty_like(h)
    rstd = torch.empty(rows, device="cuda"); dg = torch.empty(cols, device="cuda")
    M.rmsnorm_residual_fwd(x, res, gamma, h, y, rstd, EPS_N)
    M.rmsnorm_residual_bwd(dy, None, x, res, gamma, rstd, dx, dg, EPS_N,
                           M.workspace(M.OP_RMSNORM_RESIDUAL_BWD, rows, 0, cols))
    torch.cuda.synchronize()
    idx = np.unique(np.concatenate([[0, rows - 1], np.random.Generator(np.random.PCG64(5)).choice(rows, 64, replace=False)]))
    g = inp["gamma"].astype(np.float64)
    f = orc.rmsnorm_residual_fwd(_f64(inp["x"][idx]), _f64(inp["res"][idx]), g, EPS_N)
    b = orc.rmsnorm_residual_bwd(_f64(inp["dy"][idx]), None, _f64(inp["x"][idx]),
                                 _f64(inp["res"][idx]), g, EPS_N)
    ti = torch.from_numpy(idx).cuda()
    err_bf16(y[ti], f["y"])
    err_bf16(dx[ti], b["dx"])
    # dgamma over all rows, checked against the oracle in full
    full = orc.rmsnorm_residual_bwd(_f64(inp["dy"]), None, _f64(inp["x"]), _f64(inp["res"]), g,
                                    EPS_N)
    err_grad(dg, full["dgamma"])


# ---------------------------------------------------------------------------
# aggregate + weighted RMSNorm
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,n,C", [(1, 4, 8), (129, 4, 264), (67, 8, 64), (200, 8, 7168),
                                   (300, 4, 4096)])
@pytest.mark.parametrize("with_dy", [True, False])
def test_aggregate_rmsnorm(M, orc, T, n, C, with_dy):
    inp = mi.layer_inputs(T, n, C, 400 + T + C, grads=True)
    nin = mi.norm_inputs(T, C, 401 + T)
    H = mi.gate_inputs(T, n, 402 + T)["H_pre"]
    x, Hd, gamma = dev_bf16(inp["x"]), dev_f32(H), dev_f32(nin["gamma"])
    dyn, dy = dev_bf16(nin["dy"]), dev_bf16(inp["dy"]) if with_dy else None
    by, y = canary((T, C), torch.bfloat16)
    byn, yn = canary((T, C), torch.bfloat16)
    br, rstd = canary((T,), torch.float32)
    bdx, dx = canary((T, n, C), torch.bfloat16)
    bdh, dH = canary((T, n), torch.float32)
    bg, dg = canary((C,), torch.float32)
    M.mhc_h_aggregate_rmsnorm_fwd(x, Hd, gamma, y, yn, rstd, EPS_N)
    M.mhc_h_aggregate_rmsnorm_bwd(dyn, dy, x, Hd, gamma, rstd, dx, dH, dg, EPS_N,
                                  M.workspace(M.OP_H_AGGREGATE_RMSNORM_BWD, T, n, C))
    torch.cuda.synchronize()
    for b in (by, byn, br, bdx, bdh, bg):
        check_canary(b)
    xf, g = _f64(inp["x"]), nin["gamma"].astype(np.float64)
    f = orc.h_aggregate_rmsnorm_fwd(xf, H, g, EPS_N)
    err_bf16(y, f["y"])
    err_bf16(yn, f["yn"])
    err_grad(rstd, f["rstd"], rel=1e-5)
    b = orc.h_aggregate_rmsnorm_bwd(_f64(nin["dy"]), _f64(inp["dy"]) if with_dy else None, xf, H,
                                    g, EPS_N)
    err_bf16(dx, b["dx"])
    err_grad(dH, b["dH_pre"])
    err_grad(dg, b["dgamma"])


# ---------------------------------------------------------------------------
# channel-sharded proj_rms_compute_h
# ---------------------------------------------------------------------------

def _shard_np(x, W, C, c0, c1):
    n = x.shape[1]
    xs = np.ascontiguousarray(x[:, :, c0:c1])
    Ws = np.ascontiguousarray(np.concatenate([W[i * C + c0:i * C + c1] for i in range(n)], 0))
    return xs, Ws


# "stress" draws alpha = 1, b ~ N(0, 1), W ~ N(0, 0.05), so the gates and the
# Sinkhorn leave their near-uniform regime and H is sensitive to the rounding
# of u; the 4-shard case reaches the 7B-scale K = 4096 under it.
@pytest.mark.parametrize("T,n,C,cuts,stress", [(256, 4, 256, [0, 128, 256], True),
                                               (129, 4, 264, [0, 128, 264], True),
                                               (67, 8, 136, [0, 64, 136], True),
                                               (300, 4, 1024, [0, 256, 512, 768, 1024], True),
                                               (300, 4, 1024, [0, 256, 512, 768, 1024], False)])
def test_sharded_proj_rms(M, orc, T, n, C, cuts, stress):
    O = n * n + 2 * n
    K = n * C
    if stress:
        inp = mi.layer_inputs(T, n, C, 500 + T, w_std=0.05, b_std=1.0, alpha=1.0)
    else:
        inp = mi.layer_inputs(T, n, C, 500 + T, w_std=0.02, b_std=1.0)
    dH = mi.sinkhorn_inputs(T, n, 501 + T)
    dHp = mi.gate_inputs(T, n, 502 + T)
    dH_pre, dH_post = dHp["H_pre"] - 0.5, dHp["H_pre"][:, ::-1].copy() - 0.5
    dH_res = dH["dP"]
    alpha, b = inp["alpha"], inp["b"]
    u = torch.zeros(T, O, device="cuda"); s = torch.zeros(T, device="cuda")
    shards = []
    for c0, c1 in zip(cuts[:-1], cuts[1:]):
        Cs = c1 - c0
        xs_b, Ws = _shard_np(inp["x"], inp["W"], C, c0, c1)
        xs, Wd = dev_bf16(xs_b), dev_f32(Ws)
        up = torch.empty(T, O, device="cuda"); sp = torch.empty(T, device="cuda")
        M.mhc_proj_rms_partial_fwd(xs, Wd, up, sp, M.workspace(M.OP_PROJ_RMS_PARTIAL_FWD, T, n, Cs))
        u += up; s += sp  # the all-reduce over shards
        shards.append((c0, c1, xs, Wd))
    Hpre = torch.empty(T, n, device="cuda"); Hpost = torch.empty(T, n, device="cuda")
    Hres = torch.empty(T, n, n, device="cuda"); r = torch.empty(T, device="cuda")
    M.mhc_compute_h_fwd(u, s, K, dev_f32(alpha), dev_f32(b), ITERS, EPS_SK, EPS_RMS, Hpre, Hpost,
                        Hres, r)
    du = torch.empty(T, O, device="cuda"); coef = torch.empty(T, device="cuda")
    dalpha = torch.empty(3, device="cuda"); db = torch.empty(O, device="cuda")
    M.mhc_compute_h_bwd(dev_f32(dH_pre), dev_f32(dH_post), dev_f32(dH_res), u, s, K,
                        dev_f32(alpha), dev_f32(b), ITERS, EPS_SK, EPS_RMS, du, coef, dalpha, db,
                        M.workspace(M.OP_COMPUTE_H_BWD, T, n, 8))
    dx = torch.empty(T, n, C, dtype=torch.bfloat16, device="cuda")
    dW = torch.empty(K, O, device="cuda")
    for c0, c1, xs, Wd in shards:
        Cs = c1 - c0
        dxs = torch.empty(T, n, Cs, dtype=torch.bfloat16, device="cuda")
        dWs = torch.empty(n * Cs, O, device="cuda")
        M.mhc_proj_rms_partial_bwd(xs, Wd, du, coef, dxs, dWs,
                                   M.workspace(M.OP_PROJ_RMS_PARTIAL_BWD, T, n, Cs))
        dx[:, :, c0:c1] = dxs
        for i in range(n):
            dW[i * C + c0:i * C + c1] = dWs[i * Cs:(i + 1) * Cs]
    torch.cuda.synchronize()
    xf = _f64(inp["x"])
    ref = orc.proj_rms_compute_h_fwd(xf, inp["W"], alpha, b, n, ITERS, EPS_SK, EPS_RMS)
    err_h(Hpre, ref["H_pre"]); err_h(Hpost, ref["H_post"]); err_h(Hres, ref["H_res"])
    err_grad(u, ref["u"])
    err_grad(r, ref["r"], rel=1e-5)
    sref = np.sum(xf.reshape(T, -1) ** 2, axis=1)
    err_grad(s, sref, rel=1e-5)
    cb = orc.compute_h_bwd_from_sums(dH_pre, dH_post, dH_res, ref["u"], sref, K, alpha, b, n,
                                     ITERS, EPS_SK, EPS_RMS)
    err_grad(du, cb["du"])
    err_grad(coef, cb["coef"])
    err_grad(dalpha, cb["dalpha"])
    err_grad(db, cb["db"])
    rb = orc.proj_rms_compute_h_bwd(dH_pre, dH_post, dH_res, xf, inp["W"], alpha, b, n, ITERS,
                                    EPS_SK, EPS_RMS)
    err_bf16(dx, rb["dx"])
    err_grad(dW, rb["dW"])


# ---------------------------------------------------------------------------
# batch-invariant mode (RL-Kernel PR #383: fixed-K / batch-invariant GEMM)
# ---------------------------------------------------------------------------

def _layer_on(M, t, T, n, C):
    from tests.test_gpu_ops import run_layer
    return run_layer(M, t, T, n, C)


@pytest.mark.parametrize("n,C", [(4, 1024), (8, 512)])
def test_batch_invariant_mode(M, n, C):
    """With the mode on, the outputs of a token do not depend on the batch it
    is in: 64 tokens alone and the same 64 tokens at offset 517 of a
    1000-token batch give bitwise equal per-token outputs, forward and
    backward."""
    big = mi.layer_inputs(1000, n, C, 600, w_std=0.02, b_std=1.0, alpha=1.0)
    off, Ts = 517, 64
    small = dict(big)
    for k in ("x", "f", "dout", "dy"):
        small[k] = np.ascontiguousarray(big[k][off:off + Ts])
    M.mhc_set_batch_invariant(True)
    try:
        assert M.mhc_batch_invariant()
        ob = _layer_on(M, big, 1000, n, C)
        os_ = _layer_on(M, small, Ts, n, C)
    finally:
        M.mhc_set_batch_invariant(False)
    for k in ("H_pre", "H_post", "H_res", "u", "r", "y", "out", "dx", "df"):
        a, b = host(ob[k][off:off + Ts]), host(os_[k])
        assert np.array_equal(a, b), f"{k} depends on the batch"


# ---------------------------------------------------------------------------
# cross-layer fusion: the post-mix of layer l with layer l+1's proj_rms pass
# ---------------------------------------------------------------------------

def _post_proj_inputs(T, n, C, seed, alpha=(0.5, 0.8, 1.0), w_std=0.02):
    inp = mi.layer_inputs(T, n, C, seed, grads=False)
    g = np.random.Generator(np.random.PCG64(seed + 1))
    O = n * n + 2 * n
    return {"res": inp["x"], "f": inp["f"], "bias": inp["bias"],
            "Hres": g.random((T, n, n), dtype=np.float32),
            "Hpost": (2.0 * g.random((T, n), dtype=np.float32)).astype(np.float32),
            "W2": (w_std * g.standard_normal((n * C, O), dtype=np.float32)).astype(np.float32),
            "a2": np.asarray(alpha, dtype=np.float32),
            "b2": g.standard_normal(O, dtype=np.float32)}


def _run_post_proj(M, p, T, n, C):
    O = n * n + 2 * n
    d = {"res": dev_bf16(p["res"]), "f": dev_bf16(p["f"]),
         "bias": None if p["bias"] is None else dev_bf16(p["bias"]),
         "Hres": dev_f32(p["Hres"]), "Hpost": dev_f32(p["Hpost"]), "W2": dev_f32(p["W2"]),
         "a2": dev_f32(p["a2"]), "b2": dev_f32(p["b2"])}
    bufs, o = {}, {}
    for k, shape, dt in (("out", (T, n, C), torch.bfloat16), ("H_pre", (T, n), torch.float32),
                         ("H_post", (T, n), torch.float32), ("H_res", (T, n, n), torch.float32),
                         ("u", (T, O), torch.float32), ("r", (T,), torch.float32)):
        bufs[k], o[k] = canary(shape, dt)
    ws = M.workspace(M.OP_H_POST_BDA_COMPUTE_H_FWD, T, n, C)
    M.mhc_h_post_bda_compute_h_fwd(d["res"], d["f"], d["bias"], d["Hres"], d["Hpost"], d["W2"],
                                   d["a2"], d["b2"], ITERS, EPS_SK, EPS_RMS, o["out"], o["H_pre"],
                                   o["H_post"], o["H_res"], o["u"], o["r"], ws)
    return d, bufs, o


# (2500, 8, 1032): 20 token tiles x 7 splits of ten 16-channel stages (ragged
# last split, last stage half past C), so both x-stage and W-stage rings wrap
# and the out.W'_hi buffers are drained five times per CTA
@pytest.mark.parametrize("T,n,C", [(1, 4, 64), (256, 4, 256), (300, 4, 264), (129, 4, 520),
                                   (67, 8, 64), (200, 8, 136), (2500, 8, 1032)])
def test_post_bda_compute_h_fused(M, orc, T, n, C):
    """The fused op against the two ops run one after the other (out bitwise
    equal; the next layer's H from the same bf16 out, equal up to the order of
    the fp32 sums) and against the oracle composition."""
    p = _post_proj_inputs(T, n, C, 700 + T + C)
    d, bufs, o = _run_post_proj(M, p, T, n, C)
    out_sep = torch.empty_like(o["out"])
    M.mhc_h_post_bda_fwd(d["res"], d["f"], d["bias"], d["Hres"], d["Hpost"], out_sep)
    sep = {k: torch.empty_like(o[k]) for k in ("H_pre", "H_post", "H_res", "u", "r")}
    M.mhc_proj_rms_compute_h_fwd(out_sep, d["W2"], d["a2"], d["b2"], ITERS, EPS_SK, EPS_RMS,
                                 sep["H_pre"], sep["H_post"], sep["H_res"], sep["u"], sep["r"],
                                 M.workspace(M.OP_PROJ_RMS_COMPUTE_H_FWD, T, n, C))
    torch.cuda.synchronize()
    for b in bufs.values():
        check_canary(b)
    assert torch.equal(o["out"], out_sep), "fused out differs from h_post_bda"
    for k in ("H_pre", "H_post", "H_res"):
        assert float((o[k] - sep[k]).abs().max()) <= 2e-6, k
    _check_post_proj(orc, p, o, n, slice(None))


def _check_post_proj(orc, p, o, n, idx):
    """Two checks.

    1. Against the oracle's own composition (h_post_bda_compute_h_fwd: the
       fp64 post-mix, rounded by the oracle's bf16_rne, then the next
       layer's proj_rms_compute_h).  The bf16 rounding of out is a
       quantisation decision: where the exact sum lies next to a rounding
       midpoint the kernel's fp32 sum may round the other way (one bf16 ulp),
       and with alpha near 1 that moves that token's H by ~1e-4.  So: the
       elements of the stored out that differ from the oracle's rounded out
       are counted (a small fraction: an fp32 sum lands that close to a
       midpoint about once in 1e4 elements; each at most one bf16 ulp
       apart), and H, u, r meet their tolerances on every token without
       such an element.
    2. The next layer's H, u, r against the oracle's proj_rms_compute_h of
       the out the kernel stored (the decision taken in the kernel's
       precision, as the next layer sees it), on every token."""
    ti = torch.from_numpy(np.arange(o["out"].shape[0])[idx]).cuda()
    Tn = int(ti.numel())
    res = p["res"][idx]
    C = p["res"].shape[2]
    bias64 = np.zeros(C) if p["bias"] is None else _f64(p["bias"])
    comp = orc.h_post_bda_compute_h_fwd(_f64(res), _f64(p["f"][idx]), bias64,
                                        p["Hres"][idx], p["Hpost"][idx], p["W2"], p["a2"],
                                        p["b2"], n, ITERS, EPS_SK, EPS_RMS)
    out_k = host(o["out"][ti])
    err_bf16(out_k, comp["out"])
    # 1: the oracle's composition
    xr = comp["x_next"].reshape(Tn, -1)
    diff = out_k.reshape(Tn, -1) != xr
    flipped = np.any(diff, axis=1)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(xr), 2.0 ** -126))) - 7)
    # where the post-mix cancels, the fp32 sum's own rounding (a few 2^-24 of
    # the sum of the terms' magnitudes) can exceed one ulp of the result
    terms = (np.abs(p["Hpost"][idx])[:, :, None] * np.abs(_f64(p["f"][idx]) + bias64)[:, None, :]
             + np.einsum("tji,tjc->tic", np.abs(p["Hres"][idx]).astype(np.float64), np.abs(_f64(res))))
    slack = np.maximum(ulp, 2.0 ** -20 * terms.reshape(Tn, -1))
    assert np.all(np.abs(out_k.reshape(Tn, -1) - xr)[diff] <= slack[diff]), \
        "stored out differs from the oracle's rounding by more than one bf16 ulp"
    nflip = int(diff.sum())
    assert nflip <= max(4, diff.size // 1000), f"{nflip} of {diff.size} elements rounded apart"
    keep = ~flipped
    for k in ("H_pre", "H_post", "H_res"):
        err_h(host(o[k][ti])[keep], comp[k][keep])
    err_grad(host(o["u"][ti])[keep], comp["u"][keep])
    err_grad(host(o["r"][ti])[keep], comp["r"][keep])
    # 2: the oracle's second stage on the out the kernel stored
    h = orc.proj_rms_compute_h_fwd(out_k, p["W2"], p["a2"], p["b2"], n, ITERS, EPS_SK, EPS_RMS)
    for k in ("H_pre", "H_post", "H_res"):
        err_h(o[k][ti], h[k])
    err_grad(o["u"][ti], h["u"])
    err_grad(o["r"][ti], h["r"])


def test_post_bda_compute_h_fused_7b_sampled(M, orc):
    """Full 7B-scale shape (T=16384, n=4, C=4096, 64 channel blocks of 128
    token tiles); the oracle recomputes a sample of tokens (all per-token)."""
    T, n, C = 16384, 4, 4096
    p = _post_proj_inputs(T, n, C, 3, alpha=(0.01, 0.01, 0.01))
    _, bufs, o = _run_post_proj(M, p, T, n, C)
    torch.cuda.synchronize()
    for b in bufs.values():
        check_canary(b)
    g = np.random.Generator(np.random.PCG64(9))
    idx = np.unique(np.concatenate([[0, 127, 128, T - 1], g.choice(T, 40, replace=False)]))
    _check_post_proj(orc, p, o, n, idx)


@pytest.mark.parametrize("T,n,C", [(130, 4, 96), (1, 8, 16), (300, 8, 264)])
def test_post_bda_compute_h_fused_no_bias(M, orc, T, n, C):
    """bias = NULL (the n = 8 kernel then loads no bias box); one token at
    n = 8; against the two ops run one after the other and the oracle."""
    p = _post_proj_inputs(T, n, C, 900 + T + C)
    p["bias"] = None
    d, bufs, o = _run_post_proj(M, p, T, n, C)
    out_sep = torch.empty_like(o["out"])
    M.mhc_h_post_bda_fwd(d["res"], d["f"], None, d["Hres"], d["Hpost"], out_sep)
    torch.cuda.synchronize()
    for b in bufs.values():
        check_canary(b)
    assert torch.equal(o["out"], out_sep), "fused out differs from h_post_bda"
    _check_post_proj(orc, p, o, n, slice(None))


def test_post_bda_compute_h_fused_n8_sampled(M, orc):
    """n = 8 at C = 7168 (448 channel blocks; 32 token tiles x 4 splits of 112
    stages each); the oracle recomputes a sample of tokens."""
    T, n, C = 4096, 8, 7168
    p = _post_proj_inputs(T, n, C, 5, alpha=(0.01, 0.01, 0.01))
    _, bufs, o = _run_post_proj(M, p, T, n, C)
    torch.cuda.synchronize()
    for b in bufs.values():
        check_canary(b)
    g = np.random.Generator(np.random.PCG64(11))
    idx = np.unique(np.concatenate([[0, 127, 128, T - 1], g.choice(T, 24, replace=False)]))
    _check_post_proj(orc, p, o, n, idx)


@pytest.mark.parametrize("n", [4, 8])
def test_post_bda_compute_h_fused_batch_invariant(M, n):
    """Batch-invariant mode covers the fused op: 64 tokens alone and at
    offset 517 of a 1000-token batch give bitwise equal outputs."""
    C = 1024
    big = _post_proj_inputs(1000, n, C, 640)
    off, Ts = 517, 64
    small = dict(big)
    for k in ("res", "f", "Hres", "Hpost"):
        small[k] = np.ascontiguousarray(big[k][off:off + Ts])
    M.mhc_set_batch_invariant(True)
    try:
        _, _, ob = _run_post_proj(M, big, 1000, n, C)
        _, _, os_ = _run_post_proj(M, small, Ts, n, C)
        torch.cuda.synchronize()
    finally:
        M.mhc_set_batch_invariant(False)
    for k in ("out", "H_pre", "H_post", "H_res", "u", "r"):
        assert torch.equal(ob[k][off:off + Ts], os_[k]), f"{k} depends on the batch"
