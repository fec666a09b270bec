"""Pins for the fp64 oracle: checks against facts that do not come from it.

Each test ties one oracle function to something fixed outside the oracle:
a hand-worked example (tests/golden), a closed form, an invariant of the
mathematics, a library routine (numpy einsum/matmul, torch rms_norm), central
finite differences of the oracle's own forward, or a torch autograd graph of
the forward.  A dropped term, a wrong sign or index, or a transposed operand
in the oracle breaks at least one of them.

Definitions: rwkv-ops mhu_ffi.cu FFI handlers (Sinkhorn, RMSNorm, stream
aggregate, post op), Megatron-Core core.fusions.fused_mhc_kernels (fused_
sinkhorn, fused_h_aggregate, fused_h_post_bda "H_res.T @ residual + H_post *
(x + bias)", fused_proj_rms_compute_h), RL-Kernel PR #383 (fp32_gemm_rms RMS
backward with the zero-row guard; three alpha scalars over PRE/POST/COMB).
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _sig(z):
    return 1.0 / (1.0 + np.exp(-z))


def _assert_fd(fd, an, rtol=1e-4, atol=1e-8):
    fd, an = np.asarray(fd), np.asarray(an)
    scale = max(float(np.max(np.abs(an))), 1e-12)
    err = float(np.max(np.abs(fd - an)))
    assert err <= rtol * scale + atol, f"fd mismatch: err {err:.3e} scale {scale:.3e}"


# ----------------------------------------------------------------------------
# Sinkhorn
# ----------------------------------------------------------------------------

def test_sinkhorn_hand_worked_golden(orc):
    """tests/golden/sinkhorn_hand_worked.txt: exact rational answers."""
    path = os.path.join(GOLDEN, "sinkhorn_hand_worked.txt")
    cases = 0
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        lhs, rhs = line.split("|")
        toks = lhs.split()
        n = int(toks[1])
        E = np.array([float(v) for v in toks[2:]]).reshape(n, n)
        P_exp = np.array([float(Fraction(v)) for v in rhs.split()]).reshape(n, n)
        P = orc.sinkhorn_fwd(np.log(E), 1, 0.0)
        np.testing.assert_allclose(P, P_exp, rtol=0, atol=1e-15)
        cases += 1
    assert cases == 2


@pytest.mark.parametrize("n", [2, 4, 8])
def test_sinkhorn_rank1_is_uniform_after_one_iteration(orc, n):
    """z[i,j] = a_i + b_j: exp(z) is rank one, one row+column pass gives J/n."""
    rng = _rng(11)
    a, b = rng.normal(size=n), rng.normal(size=n)
    z = a[:, None] + b[None, :]
    P = orc.sinkhorn_fwd(z, 1, 0.0)
    np.testing.assert_allclose(P, np.full((n, n), 1.0 / n), rtol=0, atol=1e-15)


@pytest.mark.parametrize("n", [4, 8])
def test_sinkhorn_doubly_stochastic_fixed_point(orc, n):
    """z = log P for a doubly stochastic P (Birkhoff mix of permutations)."""
    rng = _rng(12)
    P = np.zeros((n, n))
    w = rng.uniform(0.1, 1.0, size=5)
    w /= w.sum()
    for wk in w:
        P[np.arange(n), rng.permutation(n)] += wk
    P += 1e-3
    P /= P.sum(1, keepdims=True)  # rows sum 1 ...
    P /= P.sum(0, keepdims=True)  # ... columns 1; repeat to convergence
    for _ in range(200):
        P /= P.sum(1, keepdims=True)
        P /= P.sum(0, keepdims=True)
    out = orc.sinkhorn_fwd(np.log(P), 20, 0.0)
    np.testing.assert_allclose(out, P, rtol=0, atol=1e-12)


@pytest.mark.parametrize("n", [4, 8])
def test_sinkhorn_permutation_limit(orc, n):
    """A large multiple of a permutation's indicator tends to that permutation."""
    perm = _rng(13).permutation(n)
    Pm = np.zeros((n, n))
    Pm[np.arange(n), perm] = 1.0
    out = orc.sinkhorn_fwd(40.0 * Pm, 20, 0.0)
    np.testing.assert_allclose(out, Pm, rtol=0, atol=1e-12)


def test_sinkhorn_zero_iterations_is_exp(orc):
    z = _rng(14).normal(size=(3, 4, 4))
    np.testing.assert_allclose(orc.sinkhorn_fwd(z, 0, 1e-6), np.exp(z), rtol=1e-15)


@pytest.mark.parametrize("n", [4, 8])
def test_sinkhorn_sums_and_sign(orc, n):
    """Nonnegative; after a column step the column sums are c/(c+eps)."""
    eps = 1e-6
    z = _rng(15).normal(scale=0.5, size=(256, n, n))
    P = orc.sinkhorn_fwd(z, 20, eps)
    assert np.all(P >= 0.0)
    # columns: 1 - eps within 1e-6 (the last step divides each column by sum+eps)
    assert np.max(np.abs(P.sum(1) - (1.0 - eps))) <= 1e-6
    # rows: converged to within 1e-6 of the same value for these logits
    assert np.max(np.abs(P.sum(2) - (1.0 - eps))) <= 1e-6


def test_sinkhorn_step_order_row_first(orc):
    """One iteration on a non-rank-one matrix: row step then column step."""
    E = np.array([[1.0, 2.0], [3.0, 4.0]])
    P = orc.sinkhorn_fwd(np.log(E), 1, 0.0)
    # column-first would give [[1/4... ]] with rows summing to 1 instead
    assert abs(P[:, 0].sum() - 1.0) < 1e-15 and abs(P[0].sum() - 1.0) > 1e-3


@pytest.mark.parametrize("n,eps", [(4, 1e-6), (8, 1e-6), (4, 0.3)])
def test_sinkhorn_bwd_finite_differences(orc, n, eps):
    rng = _rng(16)
    z = rng.normal(size=(3, n, n))
    g = rng.normal(size=(3, n, n))
    iters = 20
    an = orc.sinkhorn_bwd(g, z, iters, eps)
    h = 1e-6
    fd = np.zeros_like(z)
    for idx in np.ndindex(z.shape):
        zp, zm = z.copy(), z.copy()
        zp[idx] += h
        zm[idx] -= h
        m = idx[0]
        fd[idx] = (np.sum(g[m] * orc.sinkhorn_fwd(zp[m], iters, eps))
                   - np.sum(g[m] * orc.sinkhorn_fwd(zm[m], iters, eps))) / (2 * h)
    _assert_fd(fd, an)


@pytest.mark.parametrize("n", [4, 8])
def test_sinkhorn_bwd_row_shift_invariance(orc, n):
    """eps = 0: the first row step cancels a constant added to a row of z."""
    rng = _rng(17)
    z = rng.normal(size=(16, n, n))
    g = rng.normal(size=(16, n, n))
    d = orc.sinkhorn_bwd(g, z, 20, 0.0)
    assert np.max(np.abs(d.sum(2))) < 1e-12 * max(1.0, np.max(np.abs(d)))


def _torch_sinkhorn(z, iters, eps):
    A = torch.exp(z)
    for _ in range(iters):
        A = A / (A.sum(-1, keepdim=True) + eps)
        A = A / (A.sum(-2, keepdim=True) + eps)
    return A


@pytest.mark.parametrize("n", [4, 8])
def test_sinkhorn_bwd_matches_autograd(orc, n):
    rng = _rng(18)
    z = rng.normal(size=(32, n, n))
    g = rng.normal(size=(32, n, n))
    zt = torch.tensor(z, dtype=torch.float64, requires_grad=True)
    (_torch_sinkhorn(zt, 20, 1e-6) * torch.tensor(g)).sum().backward()
    np.testing.assert_allclose(orc.sinkhorn_bwd(g, z, 20, 1e-6), zt.grad.numpy(),
                               rtol=1e-9, atol=1e-12)


# ----------------------------------------------------------------------------
# h_aggregate
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("n", [4, 8])
def test_aggregate_one_hot_selects_stream(orc, n):
    from mhc_inputs import bf16_bits, bf16_bits_to_f32
    rng = _rng(20)
    T, C = 5, 24
    x = bf16_bits(rng.standard_normal((T, n, C), dtype=np.float32))
    sel = rng.integers(0, n, size=T)
    H = np.zeros((T, n))
    H[np.arange(T), sel] = 1.0
    y = orc.h_aggregate_fwd(x, H)
    xf = bf16_bits_to_f32(x)
    np.testing.assert_array_equal(y, xf[np.arange(T), sel].astype(np.float64))


def test_aggregate_matches_einsum_and_bwd(orc):
    rng = _rng(21)
    T, n, C = 6, 4, 16
    x = rng.normal(size=(T, n, C))
    H = rng.uniform(size=(T, n))
    dy = rng.normal(size=(T, C))
    np.testing.assert_allclose(orc.h_aggregate_fwd(x, H), np.einsum("ti,tic->tc", H, x),
                               rtol=1e-14, atol=1e-14)
    b = orc.h_aggregate_bwd(dy, x, H)
    np.testing.assert_allclose(b["dx"], np.einsum("ti,tc->tic", H, dy), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(b["dH_pre"], np.einsum("tc,tic->ti", dy, x), rtol=1e-13,
                               atol=1e-13)


# ----------------------------------------------------------------------------
# h_post_bda
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("n", [4, 8])
def test_post_bda_identity_copies_residual(orc, n):
    from mhc_inputs import bf16_bits, bf16_bits_to_f32
    rng = _rng(30)
    T, C = 4, 32
    x = bf16_bits(rng.standard_normal((T, n, C), dtype=np.float32))
    f = bf16_bits(rng.standard_normal((T, C), dtype=np.float32))
    bias = bf16_bits(rng.standard_normal((C,), dtype=np.float32))
    Hres = np.broadcast_to(np.eye(n), (T, n, n)).copy()
    out = orc.h_post_bda_fwd(x, f, bias, Hres, np.zeros((T, n)))
    np.testing.assert_array_equal(out, bf16_bits_to_f32(x).astype(np.float64))


def test_post_bda_permutation_and_bias_branch(orc):
    from mhc_inputs import bf16_bits_to_f32, bf16_bits
    rng = _rng(31)
    T, n, C = 3, 4, 8
    x = bf16_bits(rng.standard_normal((T, n, C), dtype=np.float32))
    f = bf16_bits(rng.standard_normal((T, C), dtype=np.float32))
    bias = bf16_bits(rng.standard_normal((C,), dtype=np.float32))
    xf = bf16_bits_to_f32(x).astype(np.float64)
    perm = np.array([2, 0, 3, 1])
    Hres = np.zeros((T, n, n))
    Hres[:, np.arange(n), perm] = 1.0  # residual stream j goes to output perm[j]
    out = orc.h_post_bda_fwd(x, f, bias, Hres, np.zeros((T, n)))
    np.testing.assert_array_equal(out[:, perm], xf)
    out2 = orc.h_post_bda_fwd(x, f, bias, np.zeros((T, n, n)), np.ones((T, n)))
    fb = bf16_bits_to_f32(f).astype(np.float64) + bf16_bits_to_f32(bias).astype(np.float64)
    np.testing.assert_array_equal(out2, np.broadcast_to(fb[:, None, :], (T, n, C)))


def test_post_bda_matches_einsum(orc):
    rng = _rng(32)
    T, n, C = 3, 8, 8
    x, f, bias = rng.normal(size=(T, n, C)), rng.normal(size=(T, C)), rng.normal(size=C)
    Hres, Hpost = rng.uniform(size=(T, n, n)), rng.uniform(size=(T, n))
    dout = rng.normal(size=(T, n, C))
    ref = np.einsum("tji,tjc->tic", Hres, x) + Hpost[:, :, None] * (f + bias)[:, None, :]
    np.testing.assert_allclose(orc.h_post_bda_fwd(x, f, bias, Hres, Hpost), ref, rtol=1e-13,
                               atol=1e-13)
    b = orc.h_post_bda_bwd(dout, x, f, bias, Hres, Hpost)
    np.testing.assert_allclose(b["dres"], np.einsum("tji,tic->tjc", Hres, dout), atol=1e-13)
    np.testing.assert_allclose(b["dH_res"], np.einsum("tjc,tic->tji", x, dout), atol=1e-12)
    np.testing.assert_allclose(b["dH_post"], np.einsum("tic,tc->ti", dout, f + bias),
                               atol=1e-12)
    np.testing.assert_allclose(b["df"], np.einsum("ti,tic->tc", Hpost, dout), atol=1e-13)
    np.testing.assert_allclose(b["dbias"], np.einsum("ti,tic->c", Hpost, dout), atol=1e-12)


def test_post_bda_bwd_finite_differences(orc):
    rng = _rng(33)
    T, n, C = 2, 4, 4
    x, f, bias = rng.normal(size=(T, n, C)), rng.normal(size=(T, C)), rng.normal(size=C)
    Hres, Hpost = rng.uniform(size=(T, n, n)), rng.uniform(size=(T, n))
    dout = rng.normal(size=(T, n, C))

    def L(x_, f_, b_, Hr, Hp):
        return float(np.sum(dout * orc.h_post_bda_fwd(x_, f_, b_, Hr, Hp)))

    an = orc.h_post_bda_bwd(dout, x, f, bias, Hres, Hpost)
    h = 1e-6
    for name, arr, key in [("x", x, "dres"), ("f", f, "df"), ("bias", bias, "dbias"),
                           ("Hres", Hres, "dH_res"), ("Hpost", Hpost, "dH_post")]:
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            args = {"x": x, "f": f, "bias": bias, "Hres": Hres, "Hpost": Hpost}
            p, m = arr.copy(), arr.copy()
            p[idx] += h
            m[idx] -= h
            args[name] = p
            lp = L(args["x"], args["f"], args["bias"], args["Hres"], args["Hpost"])
            args[name] = m
            lm = L(args["x"], args["f"], args["bias"], args["Hres"], args["Hpost"])
            fd[idx] = (lp - lm) / (2 * h)
        _assert_fd(fd, an[key])


# ----------------------------------------------------------------------------
# proj_rms_compute_h
# ----------------------------------------------------------------------------

def _proj_case(seed, T=3, n=4, C=8, alpha=(0.7, 1.1, 0.9), w_std=0.3):
    rng = _rng(seed)
    O = n * n + 2 * n
    return dict(x=rng.normal(size=(T, n, C)), W=rng.normal(scale=w_std, size=(n * C, O)),
                alpha=np.array(alpha), b=rng.normal(size=O), n=n)


@pytest.mark.parametrize("n", [4, 8])
def test_proj_matches_numpy_matmul_and_gates(orc, n):
    c = _proj_case(40, T=5, n=n, C=16)
    T, K = 5, n * 16
    eps_rms, eps_sk, iters = 1e-6, 1e-6, 20
    out = orc.proj_rms_compute_h_fwd(c["x"], c["W"], c["alpha"], c["b"], n, iters, eps_sk,
                                     eps_rms)
    xf = c["x"].reshape(T, K)
    u = xf @ c["W"]
    r = 1.0 / (np.sqrt(np.mean(xf * xf, axis=1)) + eps_rms)
    np.testing.assert_allclose(out["u"], u, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["r"], r, rtol=1e-14)
    a = np.concatenate([np.full(n, c["alpha"][0]), np.full(n, c["alpha"][1]),
                        np.full(n * n, c["alpha"][2])])
    z = a[None] * r[:, None] * u + c["b"][None]
    np.testing.assert_allclose(out["H_pre"], _sig(z[:, :n]), rtol=1e-12)
    np.testing.assert_allclose(out["H_post"], 2.0 * _sig(z[:, n:2 * n]), rtol=1e-12)
    Hres_ref = orc.sinkhorn_fwd(z[:, 2 * n:].reshape(T, n, n), iters, eps_sk)
    np.testing.assert_allclose(out["H_res"], Hres_ref, rtol=1e-12)


def test_proj_zero_weight_closed_form(orc):
    """W = 0 gives z = b for every token: H depends on b alone."""
    n = 4
    c = _proj_case(41, T=4, n=n)
    W0 = np.zeros_like(c["W"])
    out = orc.proj_rms_compute_h_fwd(c["x"], W0, c["alpha"], c["b"], n, 20, 1e-6, 1e-6)
    b = c["b"]
    np.testing.assert_array_equal(out["H_pre"], np.broadcast_to(_sig(b[:n]), (4, n)))
    np.testing.assert_array_equal(out["H_post"], np.broadcast_to(2 * _sig(b[n:2 * n]), (4, n)))
    ref = orc.sinkhorn_fwd(b[2 * n:].reshape(n, n), 20, 1e-6)
    np.testing.assert_array_equal(out["H_res"], np.broadcast_to(ref, (4, n, n)))


def test_proj_scale_invariance(orc):
    """Scaling x by lam leaves r*u unchanged when eps_rms = 0."""
    n = 4
    c = _proj_case(42, T=3, n=n)
    o1 = orc.proj_rms_compute_h_fwd(c["x"], c["W"], c["alpha"], c["b"], n, 20, 1e-6, 0.0)
    o2 = orc.proj_rms_compute_h_fwd(3.7 * c["x"], c["W"], c["alpha"], c["b"], n, 20, 1e-6, 0.0)
    np.testing.assert_allclose(o1["r"][:, None] * o1["u"], o2["r"][:, None] * o2["u"],
                               rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(o1["H_res"], o2["H_res"], rtol=1e-11)


def test_proj_alpha_zero_gives_no_x_or_w_grad(orc):
    n = 4
    c = _proj_case(43, T=3, n=n, alpha=(0.0, 0.0, 0.0))
    rng = _rng(44)
    dHpre, dHpost, dHres = rng.normal(size=(3, n)), rng.normal(size=(3, n)), rng.normal(size=(3, n, n))
    g = orc.proj_rms_compute_h_bwd(dHpre, dHpost, dHres, c["x"], c["W"], c["alpha"], c["b"], n,
                                   20, 1e-6, 1e-6)
    assert np.all(g["dx"] == 0.0) and np.all(g["dW"] == 0.0)
    assert np.all(np.abs(g["dalpha"]) > 0.0)


def test_proj_zero_row_is_finite_and_rms_term_vanishes(orc):
    """An all-zero token: r = 1/eps, z = b, and the RMS gradient term is 0
    (RL-Kernel PR #383 review: guard the RMS backward against a zero row)."""
    n = 4
    c = _proj_case(45, T=3, n=n)
    c["x"][1] = 0.0
    eps_rms = 1e-6
    out = orc.proj_rms_compute_h_fwd(c["x"], c["W"], c["alpha"], c["b"], n, 20, 1e-6, eps_rms)
    assert out["r"][1] == 1.0 / eps_rms
    np.testing.assert_array_equal(out["H_pre"][1], _sig(c["b"][:n]))
    rng = _rng(46)
    dHpre, dHpost, dHres = rng.normal(size=(3, n)), rng.normal(size=(3, n)), rng.normal(size=(3, n, n))
    g = orc.proj_rms_compute_h_bwd(dHpre, dHpost, dHres, c["x"], c["W"], c["alpha"], c["b"], n,
                                   20, 1e-6, eps_rms)
    assert np.all(np.isfinite(g["dx"]))
    # only the projection term remains: dx[1] lies in the span of W's columns
    O = n * n + 2 * n
    coef, *_ = np.linalg.lstsq(c["W"], g["dx"][1].reshape(-1), rcond=None)
    np.testing.assert_allclose(c["W"] @ coef, g["dx"][1].reshape(-1), atol=1e-9)
    assert coef.shape == (O,)


@pytest.mark.parametrize("n", [4, 8])
def test_proj_bwd_finite_differences(orc, n):
    T, C = 2, 4
    c = _proj_case(47, T=T, n=n, C=C)
    rng = _rng(48)
    dHpre, dHpost, dHres = rng.normal(size=(T, n)), rng.normal(size=(T, n)), rng.normal(size=(T, n, n))
    iters, eps_sk, eps_rms = 20, 1e-6, 1e-6

    def L(x, W, alpha, b):
        o = orc.proj_rms_compute_h_fwd(x, W, alpha, b, n, iters, eps_sk, eps_rms)
        return float(np.sum(dHpre * o["H_pre"]) + np.sum(dHpost * o["H_post"])
                     + np.sum(dHres * o["H_res"]))

    an = orc.proj_rms_compute_h_bwd(dHpre, dHpost, dHres, c["x"], c["W"], c["alpha"], c["b"],
                                    n, iters, eps_sk, eps_rms)
    h = 1e-6
    base = {"x": c["x"], "W": c["W"], "alpha": c["alpha"], "b": c["b"]}
    for name, key in [("x", "dx"), ("W", "dW"), ("alpha", "dalpha"), ("b", "db")]:
        arr = base[name]
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += h
            m[idx] -= h
            lp = L(**dict(base, **{name: p}))
            lm = L(**dict(base, **{name: m}))
            fd[idx] = (lp - lm) / (2 * h)
        _assert_fd(fd, an[key])


# ----------------------------------------------------------------------------
# RMSNorm (standalone)
# ----------------------------------------------------------------------------

def test_rmsnorm_matches_torch_rms_norm(orc):
    rng = _rng(50)
    x = rng.normal(size=(7, 40))
    dy = rng.normal(size=(7, 40))
    eps = 1e-6
    xt = torch.tensor(x, requires_grad=True)
    yt = torch.nn.functional.rms_norm(xt, (40,), eps=eps)
    (yt * torch.tensor(dy)).sum().backward()
    y, rstd = orc.rmsnorm_fwd(x, eps)
    np.testing.assert_allclose(y, yt.detach().numpy(), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(rstd, 1.0 / np.sqrt(np.mean(x * x, 1) + eps), rtol=1e-14)
    np.testing.assert_allclose(orc.rmsnorm_bwd(dy, x, eps), xt.grad.numpy(), rtol=1e-12,
                               atol=1e-13)


def test_rmsnorm_bwd_orthogonality(orc):
    """sum_c dx * x = rho^3 * eps * (sum_c dy x): closed form of the backward."""
    rng = _rng(51)
    x, dy, eps = rng.normal(size=(5, 12)), rng.normal(size=(5, 12)), 0.25
    dx = orc.rmsnorm_bwd(dy, x, eps)
    rho = 1.0 / np.sqrt(np.mean(x * x, 1) + eps)
    lhs = np.sum(dx * x, 1)
    rhs = rho ** 3 * eps * np.sum(dy * x, 1)
    np.testing.assert_allclose(lhs, rhs, rtol=1e-10, atol=1e-14)


# ----------------------------------------------------------------------------
# The layer: fwd composition and the three-way gradient sum
# ----------------------------------------------------------------------------

def _layer_case(seed, T=2, n=4, C=4):
    rng = _rng(seed)
    O = n * n + 2 * n
    return {"x": rng.normal(size=(T, n, C)), "f": rng.normal(size=(T, C)),
            "bias": rng.normal(size=C), "W": rng.normal(scale=0.3, size=(n * C, O)),
            "alpha": np.array([0.8, 1.2, 0.6]), "b": rng.normal(size=O),
            "dout": rng.normal(size=(T, n, C)), "dy": rng.normal(size=(T, C))}


def _torch_layer(x, f, bias, W, alpha, b, n, iters, eps_sk, eps_rms):
    T = x.shape[0]
    xf = x.reshape(T, -1)
    K = xf.shape[1]
    q = torch.sqrt((xf * xf).sum(1) / K)
    r = 1.0 / (q + eps_rms)
    u = xf @ W
    a = torch.cat([alpha[0].expand(n), alpha[1].expand(n), alpha[2].expand(n * n)])
    z = a[None] * r[:, None] * u + b[None]
    Hpre = torch.sigmoid(z[:, :n])
    Hpost = 2 * torch.sigmoid(z[:, n:2 * n])
    Hres = _torch_sinkhorn(z[:, 2 * n:].reshape(T, n, n), iters, eps_sk)
    y = torch.einsum("ti,tic->tc", Hpre, x)
    out = torch.einsum("tji,tjc->tic", Hres, x) + Hpost[:, :, None] * (f + bias)[:, None, :]
    return y, out


@pytest.mark.parametrize("n", [4, 8])
def test_layer_bwd_matches_autograd(orc, n):
    c = _layer_case(60, T=3, n=n, C=8)
    iters, eps_sk, eps_rms = 20, 1e-6, 1e-6
    fwd = orc.layer_fwd(c, n, iters, eps_sk, eps_rms)
    bwd = orc.layer_bwd(c, fwd, n, iters, eps_sk, eps_rms)
    tt = {k: torch.tensor(v, requires_grad=True) for k, v in c.items()
          if k in ("x", "f", "bias", "W", "alpha", "b")}
    y, out = _torch_layer(tt["x"], tt["f"], tt["bias"], tt["W"], tt["alpha"], tt["b"], n, iters,
                          eps_sk, eps_rms)
    np.testing.assert_allclose(fwd["y"], y.detach().numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(fwd["out"], out.detach().numpy(), rtol=1e-12, atol=1e-13)
    ((out * torch.tensor(c["dout"])).sum() + (y * torch.tensor(c["dy"])).sum()).backward()
    for ours, theirs in [("dx", "x"), ("df", "f"), ("dbias", "bias"), ("dW", "W"),
                         ("dalpha", "alpha"), ("db", "b")]:
        np.testing.assert_allclose(bwd[ours], tt[theirs].grad.numpy(), rtol=1e-9, atol=1e-11,
                                   err_msg=ours)


def test_layer_bwd_finite_differences(orc):
    n = 4
    c = _layer_case(61, T=2, n=n, C=4)
    iters, eps_sk, eps_rms = 20, 1e-6, 1e-6

    def L(cc):
        o = orc.layer_fwd(cc, n, iters, eps_sk, eps_rms)
        return float(np.sum(cc["dout"] * o["out"]) + np.sum(cc["dy"] * o["y"]))

    fwd = orc.layer_fwd(c, n, iters, eps_sk, eps_rms)
    an = orc.layer_bwd(c, fwd, n, iters, eps_sk, eps_rms)
    h = 1e-6
    for name, key in [("x", "dx"), ("f", "df"), ("bias", "dbias"), ("alpha", "dalpha"),
                      ("b", "db")]:
        arr = c[name]
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            p, m = arr.copy(), arr.copy()
            p[idx] += h
            m[idx] -= h
            fd[idx] = (L(dict(c, **{name: p})) - L(dict(c, **{name: m}))) / (2 * h)
        _assert_fd(fd, an[key])


def test_layer_no_dx_mode_matches_full(orc):
    """The reduced mode used at full size gives the same parameter grads."""
    n = 4
    c = _layer_case(62, T=4, n=n, C=8)
    fwd = orc.layer_fwd(c, n, 20, 1e-6, 1e-6)
    full = orc.layer_bwd(c, fwd, n, 20, 1e-6, 1e-6)
    red = orc.layer_bwd(c, fwd, n, 20, 1e-6, 1e-6, want_dx=False)
    for k in ("dW", "dalpha", "db", "dbias"):
        np.testing.assert_array_equal(full[k], red[k])
