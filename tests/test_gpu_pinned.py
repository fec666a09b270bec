"""GPU parity of the bit-reproducible mode (mhc_set_pinned_reductions): with
the mode on, every output of the mHC ops is bitwise equal to the fp32
pinned-order reference (oracle/mhc_oracle_pinned.c) on the same inputs.

Contract: RL-Align/RL-Kernel PR #383, PR body, "Numerical contract" (fp32;
only the four-stream tree (a0 + a1) + (a2 + a3) and a serial ascending left
fold).  The reference is pinned in tests/test_oracle_pins_pinned.py."""
import numpy as np
import pytest
import torch

import mhc_inputs as mi
from tests._util import dev_bf16, dev_f32

pytestmark = pytest.mark.gpu

ITERS, EPS_SK, EPS_RMS = mi.ITERS, mi.EPS_SK, mi.EPS_RMS


@pytest.fixture(scope="module")
def M():
    import layers_proj_rms_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return m


@pytest.fixture
def pinned(M):
    M.mhc_set_pinned_reductions(True)
    assert M.mhc_pinned_reductions()
    try:
        yield M
    finally:
        M.mhc_set_pinned_reductions(False)


def bits(t):
    """The exact bits of a tensor (bf16 as its fp32 value, fp32 as is)."""
    a = t.float().cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, np.float32)
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def same(gpu, ref, what):
    g, r = bits(gpu), bits(np.asarray(ref, np.float32))
    assert g.shape == r.shape, what
    bad = np.flatnonzero(g.ravel() != r.ravel())
    assert bad.size == 0, f"{what}: {bad.size} of {g.size} elements differ (first at {bad[0]})"


def _layer(M, inp, T, C):
    n, O = 4, 24
    t = {k: (dev_bf16(v) if v.dtype == np.uint16 else dev_f32(v)) for k, v in inp.items()
         if v is not None}
    e = lambda *s, dt=torch.float32: torch.empty(*s, dtype=dt, device="cuda")  # noqa: E731
    bf = torch.bfloat16
    o = {"H_pre": e(T, n), "H_post": e(T, n), "H_res": e(T, n, n), "u": e(T, O), "r": e(T),
         "y": e(T, C, dt=bf), "out": e(T, n, C, dt=bf), "dx": e(T, n, C, dt=bf),
         "df": e(T, C, dt=bf), "dW": e(n * C, O), "dalpha": e(3), "db": e(O), "dbias": e(C)}
    M.mhc_layer_fwd(t["x"], t["W"], t["alpha"], t["b"], t["f"], t["bias"], ITERS, EPS_SK, EPS_RMS,
                    o["H_pre"], o["H_post"], o["H_res"], o["u"], o["r"], o["y"], o["out"],
                    M.workspace(M.OP_LAYER_FWD, T, n, C))
    M.mhc_layer_bwd(t["dout"], t["dy"], t["x"], t["W"], t["alpha"], t["b"], t["f"], t["bias"],
                    o["H_pre"], o["H_post"], o["H_res"], o["u"], o["r"], ITERS, EPS_SK, EPS_RMS,
                    o["dx"], o["df"], o["dW"], o["dalpha"], o["db"], o["dbias"],
                    M.workspace(M.OP_LAYER_BWD, T, n, C))
    torch.cuda.synchronize()
    return o


@pytest.mark.parametrize("T,C,seed,stress", [(1, 8, 1, False), (37, 64, 2, False),
                                             (130, 264, 3, True), (300, 128, 4, True)])
def test_layer_bitwise(pinned, orc, T, C, seed, stress):
    kw = dict(w_std=0.05, alpha=1.0, b_std=1.0) if stress else {}
    inp = mi.layer_inputs(T, 4, C, seed, **kw)
    o = _layer(pinned, inp, T, C)
    pf = orc.pin_layer_fwd(inp, ITERS, EPS_SK, EPS_RMS)
    for k in ("H_pre", "H_post", "H_res", "u", "r", "y", "out"):
        same(o[k], pf[k], k)
    pb = orc.pin_layer_bwd(inp, pf, ITERS, EPS_SK, EPS_RMS)
    for k in ("dx", "df", "dW", "dalpha", "db", "dbias"):
        same(o[k], pb[k], k)


@pytest.mark.parametrize("T,C,seed", [(33, 72, 5), (129, 40, 6)])
def test_ops_bitwise(pinned, orc, T, C, seed):
    M = pinned
    inp = mi.layer_inputs(T, 4, C, seed, w_std=0.05, alpha=1.0, b_std=1.0)
    x, W = dev_bf16(inp["x"]), dev_f32(inp["W"])
    a, b = dev_f32(inp["alpha"]), dev_f32(inp["b"])
    e = lambda *s, dt=torch.float32: torch.empty(*s, dtype=dt, device="cuda")  # noqa: E731
    bf = torch.bfloat16
    # proj_rms_compute_h
    Hp, Hq, Hr, u, r = e(T, 4), e(T, 4), e(T, 4, 4), e(T, 24), e(T)
    M.mhc_proj_rms_compute_h_fwd(x, W, a, b, ITERS, EPS_SK, EPS_RMS, Hp, Hq, Hr, u, r,
                                 M.workspace(M.OP_PROJ_RMS_COMPUTE_H_FWD, T, 4, C))
    rng = np.random.Generator(np.random.PCG64(seed + 50))
    dHp, dHq = (rng.standard_normal((T, 4), dtype=np.float32) for _ in range(2))
    dHr = rng.standard_normal((T, 4, 4), dtype=np.float32)
    dx, dW, da, db = e(T, 4, C, dt=bf), e(4 * C, 24), e(3), e(24)
    M.mhc_proj_rms_compute_h_bwd(dev_f32(dHp), dev_f32(dHq), dev_f32(dHr), x, W, a, b, u, r,
                                 ITERS, EPS_SK, EPS_RMS, dx, dW, da, db,
                                 M.workspace(M.OP_PROJ_RMS_COMPUTE_H_BWD, T, 4, C))
    # aggregate and post-mix with the forward's H
    y = e(T, C, dt=bf)
    M.mhc_h_aggregate_fwd(x, Hp, y)
    dy = dev_bf16(inp["dy"])
    dxa, dHa = e(T, 4, C, dt=bf), e(T, 4)
    M.mhc_h_aggregate_bwd(dy, x, Hp, dxa, dHa)
    f, bias, dout = dev_bf16(inp["f"]), dev_bf16(inp["bias"]), dev_bf16(inp["dout"])
    out = e(T, 4, C, dt=bf)
    M.mhc_h_post_bda_fwd(x, f, bias, Hr, Hq, out)
    dres, dfo, dbias, dHr2, dHq2 = e(T, 4, C, dt=bf), e(T, C, dt=bf), e(C), e(T, 4, 4), e(T, 4)
    M.mhc_h_post_bda_bwd(dout, x, f, bias, Hr, Hq, dres, dfo, dbias, dHr2, dHq2,
                         M.workspace(M.OP_H_POST_BDA_BWD, T, 4, C))
    torch.cuda.synchronize()
    h = orc.pin_proj_rms_compute_h_fwd(inp["x"], inp["W"], inp["alpha"], inp["b"], ITERS, EPS_SK,
                                       EPS_RMS)
    for t_, k in ((Hp, "H_pre"), (Hq, "H_post"), (Hr, "H_res"), (u, "u"), (r, "r")):
        same(t_, h[k], k)
    g = orc.pin_proj_rms_compute_h_bwd(dHp, dHq, dHr, inp["x"], inp["W"], inp["alpha"], inp["b"],
                                       ITERS, EPS_SK, EPS_RMS)
    for t_, k in ((dx, "dx"), (dW, "dW"), (da, "dalpha"), (db, "db")):
        same(t_, g[k], "proj " + k)
    same(y, orc.pin_h_aggregate_fwd(inp["x"], h["H_pre"]), "y")
    rdx, rdH = orc.pin_h_aggregate_bwd(inp["dy"], inp["x"], h["H_pre"])
    same(dxa, rdx, "aggregate dx")
    same(dHa, rdH, "dH_pre")
    same(out, orc.pin_h_post_bda_fwd(inp["x"], inp["f"], inp["bias"], h["H_res"], h["H_post"]), "out")
    pb = orc.pin_h_post_bda_bwd(inp["dout"], inp["x"], inp["f"], inp["bias"], h["H_res"], h["H_post"])
    for t_, k in ((dres, "dres"), (dfo, "df"), (dbias, "dbias"), (dHr2, "dH_res"), (dHq2, "dH_post")):
        same(t_, pb[k], "post " + k)


def test_sinkhorn_bitwise(pinned, orc):
    M = pinned
    inp = mi.sinkhorn_inputs(1000, 4, seed=9)
    lg, dP = dev_f32(inp["logits"]), dev_f32(inp["dP"])
    P, dl = torch.empty_like(lg), torch.empty_like(lg)
    M.mhc_sinkhorn_fwd(lg, P, ITERS, EPS_SK)
    M.mhc_sinkhorn_bwd(dP, lg, dl, ITERS, EPS_SK)
    torch.cuda.synchronize()
    same(P, orc.pin_sinkhorn_fwd(inp["logits"], ITERS, EPS_SK), "P")
    same(dl, orc.pin_sinkhorn_bwd(inp["dP"], inp["logits"], ITERS, EPS_SK), "dlogits")


def test_hand_worked_trees_on_gpu(pinned):
    """The golden cases of tests/golden/pinned_trees.txt through the library:
    the four-stream tree gives 1 where the serial fold gives 0 and the exact
    sum 2, and the channel fold gives 0 where the tree would give 1."""
    M = pinned
    E24 = float(2 ** 24)
    adv = torch.tensor([E24, 1.0, 1.0, -E24], dtype=torch.bfloat16, device="cuda")
    y = torch.empty(1, 8, dtype=torch.bfloat16, device="cuda")
    x = torch.zeros(1, 4, 8, dtype=torch.bfloat16, device="cuda")
    x[0, :, 0] = adv
    M.mhc_h_aggregate_fwd(x, torch.ones(1, 4, device="cuda"), y)
    xb = torch.zeros(1, 4, 8, dtype=torch.bfloat16, device="cuda")
    xb[0, 0, :4] = adv
    dxa, dH = torch.empty_like(xb), torch.empty(1, 4, device="cuda")
    dy = torch.zeros(1, 8, dtype=torch.bfloat16, device="cuda")
    dy[0, :4] = 1.0
    M.mhc_h_aggregate_bwd(dy, xb, torch.ones(1, 4, device="cuda"), dxa, dH)
    torch.cuda.synchronize()
    assert float(y[0, 0]) == 1.0
    assert float(dH[0, 0]) == 0.0


def test_n8_refused_in_pinned_mode(pinned):
    M = pinned
    x = torch.zeros(2, 8, 8, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(2, 8, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(Exception, match="n = 4"):
        M.mhc_h_aggregate_fwd(x, torch.zeros(2, 8, device="cuda"), y)
