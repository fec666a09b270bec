"""The layer step (mhc_layer_fwd, mhc_layer_bwd, rmsnorm_fwd/bwd) captured
into one CUDA graph and replayed gives the bytes the eager calls give, also
after new inputs are copied into the captured input tensors: after its first
call an entry point puts nothing on the stream but kernel launches, so the
whole step can run as a graph (no launch gaps between kernels)."""
import numpy as np
import pytest
import torch

import mhc_inputs as mi
from tests._util import dev_bf16, dev_f32
from tests.test_gpu_ops import EPS_RMS, EPS_SK, ITERS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    import layers_proj_rms_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return m


@pytest.mark.parametrize("T,n,C", [(256, 4, 512), (200, 8, 264)])
def test_layer_step_graph_replay(M, T, n, C):
    O = n * n + 2 * n
    inp = mi.layer_inputs(T, n, C, 700 + n, rmsnorm=True)
    t = {k: (dev_bf16(v) if v.dtype == np.uint16 else dev_f32(v)) for k, v in inp.items()}
    bf = torch.bfloat16
    e = lambda *s, dt=torch.float32: torch.empty(*s, dtype=dt, device="cuda")  # noqa: E731
    o = {"H_pre": e(T, n), "H_post": e(T, n), "H_res": e(T, n, n), "u": e(T, O), "r": e(T),
         "y": e(T, C, dt=bf), "out": e(T, n, C, dt=bf), "dx": e(T, n, C, dt=bf),
         "df": e(T, C, dt=bf), "dW": e(n * C, O), "dalpha": e(3), "db": e(O), "dbias": e(C),
         "yn": e(T, C, dt=bf), "rstd": e(T), "dxn": e(T, C, dt=bf)}
    wsf = M.workspace(M.OP_LAYER_FWD, T, n, C)
    wsb = M.workspace(M.OP_LAYER_BWD, T, n, C)

    def step():
        M.mhc_layer_fwd(t["x"], t["W"], t["alpha"], t["b"], t["f"], t["bias"], ITERS, EPS_SK,
                        EPS_RMS, o["H_pre"], o["H_post"], o["H_res"], o["u"], o["r"], o["y"],
                        o["out"], wsf)
        M.mhc_layer_bwd(t["dout"], t["dy"], t["x"], t["W"], t["alpha"], t["b"], t["f"], t["bias"],
                        o["H_pre"], o["H_post"], o["H_res"], o["u"], o["r"], ITERS, EPS_SK,
                        EPS_RMS, o["dx"], o["df"], o["dW"], o["dalpha"], o["db"], o["dbias"], wsb)
        M.rmsnorm_fwd(t["x_norm"], o["yn"], o["rstd"], 1e-6)
        M.rmsnorm_bwd(t["dy_norm"], t["x_norm"], o["rstd"], o["dxn"], 1e-6)

    def snapshot():
        torch.cuda.synchronize()
        return {k: v.clone() for k, v in o.items()}

    step()
    eager = snapshot()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for k in o:
        o[k].fill_(0)
    g.replay()
    got = snapshot()
    for k in o:
        assert torch.equal(got[k], eager[k]), f"graph replay differs in {k}"
    # new inputs into the captured tensors: replay = eager on the new inputs
    inp2 = mi.layer_inputs(T, n, C, 800 + n, rmsnorm=True)
    for k, v in inp2.items():
        t[k].copy_(dev_bf16(v) if v.dtype == np.uint16 else dev_f32(v))
    g.replay()
    got2 = snapshot()
    step()
    eager2 = snapshot()
    for k in o:
        assert torch.equal(got2[k], eager2[k]), f"graph replay differs in {k} (new inputs)"
    assert not torch.equal(got2["y"], got["y"])
