"""The C ABI used from a plain C program (tests/c_client/layer_client.c: no
C++, no PyTorch; device memory from the CUDA runtime).  The program runs the
layer forward and backward on a fixed integer-pattern input and writes inputs
and outputs to a file; the same inputs through the Python binding must give
bitwise the same outputs (the same kernels), and the oracle agrees within the
tolerances."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import mhc_inputs as mi
from tests._util import dev_bf16, dev_f32, err_bf16, err_grad, err_h
from tests.test_gpu_ops import EPS_RMS, EPS_SK, ITERS, run_layer

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def M():
    import layers_proj_rms_gb300 as m
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return m


@pytest.fixture(scope="module")
def client(M, tmp_path_factory):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    libdir = os.path.dirname(M.lib_path)
    exe = str(tmp_path_factory.mktemp("c_client") / "layer_client")
    subprocess.run([cc, "-std=c99", "-O2", "-Wall", f"-I{ROOT}/include", f"-I{cuda}/include",
                    os.path.join(ROOT, "tests", "c_client", "layer_client.c"), "-o", exe,
                    os.path.join(libdir, "libmhc.so"), f"-Wl,-rpath,{libdir}",
                    f"-L{cuda}/lib64", "-lcudart", f"-Wl,-rpath,{cuda}/lib64"],
                   check=True)
    return exe


def _read(path, T, n, C):
    K, O = n * C, n * n + 2 * n
    spec = [("x", np.uint16, (T, n, C)), ("f", np.uint16, (T, C)), ("bias", np.uint16, (C,)),
            ("dout", np.uint16, (T, n, C)), ("dy", np.uint16, (T, C)),
            ("W", np.float32, (K, O)), ("alpha", np.float32, (3,)), ("b", np.float32, (O,)),
            ("H_pre", np.float32, (T, n)), ("H_post", np.float32, (T, n)),
            ("H_res", np.float32, (T, n, n)), ("u", np.float32, (T, O)), ("r", np.float32, (T,)),
            ("y", np.uint16, (T, C)), ("out", np.uint16, (T, n, C)),
            ("dx", np.uint16, (T, n, C)), ("df", np.uint16, (T, C)),
            ("dW", np.float32, (K, O)), ("dalpha", np.float32, (3,)), ("db", np.float32, (O,)),
            ("dbias", np.float32, (C,))]
    raw = open(path, "rb").read()
    d, off = {}, 0
    for name, dt, shape in spec:
        nb = int(np.prod(shape)) * np.dtype(dt).itemsize
        d[name] = np.frombuffer(raw[off:off + nb], dtype=dt).reshape(shape)
        off += nb
    assert off == len(raw)
    return d


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16) if t.dtype == torch.bfloat16 \
        else t.cpu().numpy()


@pytest.mark.parametrize("T,n,C", [(200, 4, 264), (67, 8, 64)])
def test_c_client_layer(M, orc, client, tmp_path, T, n, C):
    out_file = str(tmp_path / "layer.bin")
    r = subprocess.run([client, str(T), str(n), str(C), out_file], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    c = _read(out_file, T, n, C)
    inp = {k: c[k].copy() for k in ("x", "f", "bias", "dout", "dy", "W", "alpha", "b")}
    o = run_layer(M, inp, T, n, C)
    for k in ("H_pre", "H_post", "H_res", "u", "r", "y", "out", "dx", "df", "dW", "dalpha", "db",
              "dbias"):
        assert np.array_equal(_bits(o[k]), c[k]), f"{k} differs between the C client and Python"
    ref_f = orc.layer_fwd(inp, n, ITERS, EPS_SK, EPS_RMS)
    ref_b = orc.layer_bwd(inp, ref_f, n, ITERS, EPS_SK, EPS_RMS)
    for k in ("H_pre", "H_post", "H_res"):
        err_h(o[k], ref_f[k])
    err_bf16(o["out"], ref_f["out"])
    err_bf16(o["dx"], ref_b["dx"])
    err_grad(o["dW"], ref_b["dW"])
    err_grad(o["dbias"], ref_b["dbias"])
