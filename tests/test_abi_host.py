"""Host-only checks of the C ABI: the library loads without a GPU, exports
every symbol include/mhc.h declares, and rejects bad arguments on the host
before touching a device (no kernel is launched by these tests)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mhc.h")


@pytest.fixture(scope="module")
def L():
    from layers_proj_rms_gb300 import build as B
    B.build()
    import layers_proj_rms_gb300 as m
    return m.lib


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^MHC_API\s+[\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_op_set():
    names = set(declared_functions())
    for op in ["mhc_sinkhorn_fwd", "mhc_sinkhorn_bwd", "mhc_proj_rms_compute_h_fwd",
               "mhc_proj_rms_compute_h_bwd", "mhc_h_aggregate_fwd", "mhc_h_aggregate_bwd",
               "mhc_h_post_bda_fwd", "mhc_h_post_bda_bwd", "rmsnorm_fwd", "rmsnorm_bwd",
               "mhc_layer_fwd", "mhc_layer_bwd", "mhc_h_aggregate_static_fwd",
               "mhc_h_aggregate_static_bwd", "rmsnorm_residual_fwd", "rmsnorm_residual_bwd",
               "mhc_h_aggregate_rmsnorm_fwd", "mhc_h_aggregate_rmsnorm_bwd",
               "mhc_proj_rms_partial_fwd", "mhc_compute_h_fwd", "mhc_compute_h_bwd",
               "mhc_proj_rms_partial_bwd"]:
        assert op in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing


def test_header_compiles_as_c_and_cpp():
    """include/mhc.h is a plain C header (C99) that C++ can include too."""
    import shutil
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    hdr = os.path.join(root, "include", "mhc.h")
    for cc, lang, std in (("gcc", "c", "-std=c99"), ("g++", "c++", "-std=c++11")):
        if shutil.which(cc) is None:
            pytest.skip(f"{cc} missing")
        r = subprocess.run([cc, std, "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                            "-x", lang, hdr], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def test_status_strings_and_version(L):
    for s in range(10):
        assert L.mhc_status_string(s)
    assert L.mhc_version() >= 100


A = 0x10000  # a 16-byte-aligned fake device address; never dereferenced


def test_validation_errors_without_gpu(L):
    f = L.mhc_h_aggregate_fwd
    # unsupported n
    assert f(A, A, A, 16, 5, 64, None) == 4
    assert b"n = 5" in L.mhc_last_error()
    # C not a multiple of 8
    assert f(A, A, A, 16, 4, 60, None) == 2
    # null pointer
    assert f(None, A, A, 16, 4, 64, None) == 1
    # misaligned pointer
    assert f(A + 2, A, A, 16, 4, 64, None) == 3
    # negative T
    assert f(A, A, A, -1, 4, 64, None) == 2
    # T = 0 is a no-op and needs no pointers
    assert f(None, None, None, 0, 4, 64, None) == 0
    # all valid: reaches the device check, which fails here (no GPU)
    rc = f(A, A, A, 16, 4, 64, None)
    assert rc in (0, 8, 7)
    if rc:
        assert L.mhc_last_error()


def test_sinkhorn_iters_and_eps_checks(L):
    f = L.mhc_sinkhorn_fwd
    assert f(A, A, 10, 4, 65, ctypes.c_float(1e-6), None) == 6
    assert f(A, A, 10, 4, -1, ctypes.c_float(1e-6), None) == 6
    assert f(A, A, 10, 4, 20, ctypes.c_float(float("nan")), None) == 6
    assert f(A, A, 10, 4, 20, ctypes.c_float(-1.0), None) == 6
    assert f(A, A, 10, 6, 20, ctypes.c_float(1e-6), None) == 4


def test_workspace_sizes(L):
    ws = L.mhc_workspace_bytes
    for op in (1, 2, 3, 4, 5):
        a = ws(op, 256, 4, 256)
        b = ws(op, 16384, 4, 4096)
        assert a > 0 and b >= a and a % 256 == 0
    for op in (7, 8, 9, 10, 11, 12):
        a = ws(op, 256, 4, 256)
        b = ws(op, 16384, 4, 4096)
        assert a > 0 and b >= a and a % 256 == 0
    # the fused post-mix + next projection needs at least the projection's W_hl
    O, K = 24, 4 * 4096
    assert ws(12, 16384, 4, 4096) >= 2 * O * K * 2
    # n = 8 is fused too: its W'_hl has 3 x 80 rows of 8 C bf16
    assert ws(12, 8192, 8, 7168) >= 3 * 80 * 8 * 7168 * 2
    assert ws(12, 300, 8, 136) % 256 == 0
    # the RMSNorm op ignores n
    assert ws(6, 256, 0, 4096) == ws(6, 256, 4, 4096) > 0
    assert ws(1, 256, 5, 256) == 0
    assert ws(99, 256, 4, 256) == 0


def test_next_ops_validation_without_gpu(L):
    from layers_proj_rms_gb300 import _lib  # noqa: F401  (argtypes)
    f = L.rmsnorm_residual_fwd
    # cols not a multiple of 8; cols too large; rows = 0 is a no-op
    assert f(A, None, None, None, A, None, 4, 60, 1e-6, None) == 2
    assert f(A, None, None, None, A, None, 4, 65536, 1e-6, None) == 2
    assert f(None, None, None, None, None, None, 0, 64, 1e-6, None) == 0
    # dgamma wanted: the workspace is required
    g = L.rmsnorm_residual_bwd
    assert g(A, None, A, None, None, None, A, A, 4, 64, 1e-6, None, 0, None) == 5
    # static aggregate: dH_pre is always required
    h = L.mhc_h_aggregate_static_bwd
    assert h(A, A, A, A, None, 16, 4, 64, A, 1 << 20, None) == 1
    # fused post-mix + next projection: T = 0 is a no-op; C not a multiple
    # of 8 and a missing W_next are refused before any launch
    pp = L.mhc_h_post_bda_compute_h_fwd
    assert pp(None, None, None, None, None, None, None, None, 0, 4, 64, 20, 1e-6, 1e-6,
              None, None, None, None, None, None, None, 0, None) == 0
    assert pp(A, A, None, A, A, A, A, A, 16, 4, 60, 20, 1e-6, 1e-6,
              A, A, A, A, None, None, A, 1 << 20, None) == 2
    assert pp(A, A, None, A, A, None, A, A, 16, 4, 64, 20, 1e-6, 1e-6,
              A, A, A, A, None, None, A, 1 << 20, None) == 1
    # the tensor-core ops address rows and k = i*C + c with 32-bit TMA
    # coordinates: T or n*C of 2^31 is refused on the host
    pf = L.mhc_proj_rms_compute_h_fwd
    assert pf(A, A, A, A, 1 << 31, 4, 8, 20, 1e-6, 1e-6, A, A, A, None, None, A, 1 << 20,
              None) == 2
    assert pf(A, A, A, A, 1, 8, 1 << 28, 20, 1e-6, 1e-6, A, A, A, None, None, A, 1 << 20,
              None) == 2
    # the fault-path self-test takes 1 <= wait_us <= 1e6
    st = L.mhc_selftest_wait_timeout
    assert st(0, None) == 2 and st(2000000, None) == 2
    # compute_h needs K >= 1
    c = L.mhc_compute_h_fwd
    assert c(A, A, 0, A, A, 16, 4, 20, 1e-6, 1e-6, A, A, A, None, None) == 2


def test_workspace_checks(L):
    f = L.mhc_proj_rms_compute_h_fwd
    need = L.mhc_workspace_bytes(1, 256, 4, 256)
    args = [A, A, A, A, 256, 4, 256, 20, ctypes.c_float(1e-6), ctypes.c_float(1e-6), A, A, A,
            None, None]
    assert f(*args, A, ctypes.c_size_t(need - 1), None) == 5
    assert f(*args, None, ctypes.c_size_t(need), None) == 1
    assert f(*args, A + 16, ctypes.c_size_t(need), None) == 3


def test_layer_bwd_requires_dbias_with_bias(L):
    from layers_proj_rms_gb300 import _lib  # noqa: F401  (argtypes)
    f = L.mhc_layer_bwd
    rc = f(A, A, A, A, A, A, A, A, A, A, A, A, A, 64, 4, 64, 20, 1e-6, 1e-6, A, A, A, A, A, None,
           A, 1 << 30, None)
    assert rc == 1 and b"dbias" in L.mhc_last_error()


def test_binding_fails_loudly_without_library(tmp_path):
    """The binding never falls back: a missing libmhc.so is an ImportError."""
    import subprocess
    import sys
    code = ("import sys, os; sys.path.insert(0, %r);"
            "import layers_proj_rms_gb300._lib as L" % ROOT)
    env = dict(os.environ)
    lib = os.path.join(ROOT, "layers_proj_rms_gb300", "_build", "libmhc.so")
    hidden = lib + ".hidden_for_test"
    os.rename(lib, hidden)
    try:
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env)
    finally:
        os.rename(hidden, lib)
    assert r.returncode != 0 and "libmhc.so is missing" in r.stderr


def test_batch_invariant_mode_flag(L):
    from layers_proj_rms_gb300 import _lib  # noqa: F401  (argtypes)
    assert L.mhc_batch_invariant() == 0
    off = L.mhc_workspace_bytes(1, 256, 4, 256)
    L.mhc_set_batch_invariant(1)
    try:
        assert L.mhc_batch_invariant() == 1
        on_small = L.mhc_workspace_bytes(1, 256, 4, 256)
        on_big = L.mhc_workspace_bytes(1, 16384, 4, 256)
    finally:
        L.mhc_set_batch_invariant(0)
    # K splits fixed by K: fewer splits than the T-dependent choice at small T,
    # and the per-token part of the scratch scales with T only
    assert 0 < on_small < off
    assert on_big > on_small
