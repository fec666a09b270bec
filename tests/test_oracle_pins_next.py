"""Pins for the oracle functions of the ops beyond the layer path.

  * h_aggregate with a static H_pre [n] (rwkv-ops mhu_ffi.cu StreamAggregate
    with per_token = false);
  * rmsnorm_residual: h = x + res, y = h rho gamma, with dgamma
    (RL-Kernel PR #383 tasks P1-5 "RMSNorm + residual fork" and P1-8
    "cross-rank dgamma");
  * h_aggregate followed by the weighted RMSNorm of its output, as one op;
  * proj_rms_compute_h over channel shards (RL-Kernel PR #383 task P1-6, the
    fp32_gemm_rms TP/SP contract): partial sums, compute_h on the totals,
    per-shard backward.

As in test_oracle_pins.py each pin ties the oracle to something outside it:
numpy einsum/matmul, torch's rms_norm and its autograd, closed forms, central
finite differences, or the already-pinned layer-path oracle on the unsharded
problem (a sum over shards must give the unsharded answer).
"""
import numpy as np
import pytest
import torch

from tests.test_oracle_pins import _assert_fd, _rng


# ----------------------------------------------------------------------------
# static H_pre
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("n", [4, 8])
def test_aggregate_static_matches_einsum(orc, n):
    g = _rng(40 + n)
    T, C = 5, 24
    x = g.standard_normal((T, n, C)); H = g.random(n); dy = g.standard_normal((T, C))
    np.testing.assert_allclose(orc.h_aggregate_static_fwd(x, H), np.einsum("tic,i->tc", x, H),
                               rtol=1e-13, atol=1e-13)
    b = orc.h_aggregate_static_bwd(dy, x, H)
    np.testing.assert_allclose(b["dx"], np.einsum("i,tc->tic", H, dy), rtol=0, atol=0)
    np.testing.assert_allclose(b["dH_pre"], np.einsum("tc,tic->i", dy, x), rtol=1e-12, atol=1e-12)


def test_aggregate_static_one_hot_selects_stream(orc):
    g = _rng(47)
    x = g.standard_normal((3, 4, 16))
    for j in range(4):
        H = np.zeros(4); H[j] = 1.0
        np.testing.assert_array_equal(orc.h_aggregate_static_fwd(x, H), x[:, j, :])


def test_aggregate_static_finite_differences(orc):
    g = _rng(48)
    T, n, C = 3, 4, 8
    x = g.standard_normal((T, n, C)); H = g.random(n); dy = g.standard_normal((T, C))
    L = lambda xx, HH: float(np.sum(dy * orc.h_aggregate_static_fwd(xx, HH)))  # noqa: E731
    b = orc.h_aggregate_static_bwd(dy, x, H)
    h = 1e-6
    fd = [(L(x, H + h * e) - L(x, H - h * e)) / (2 * h) for e in np.eye(n)]
    _assert_fd(fd, b["dH_pre"])
    fdx = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        e = np.zeros_like(x); e[idx] = h
        fdx[idx] = (L(x + e, H) - L(x - e, H)) / (2 * h)
    _assert_fd(fdx, b["dx"])


# ----------------------------------------------------------------------------
# rmsnorm_residual
# ----------------------------------------------------------------------------

def _torch_rmsr(x, res, gamma, eps):
    h = x + res if res is not None else x
    return h, torch.nn.functional.rms_norm(h, (h.shape[-1],), weight=gamma, eps=eps)


@pytest.mark.parametrize("with_res,with_gamma", [(True, True), (False, True), (True, False)])
def test_rmsnorm_residual_matches_torch(orc, with_res, with_gamma):
    g = _rng(50)
    rows, cols = 6, 40
    x = g.standard_normal((rows, cols)); res = g.standard_normal((rows, cols)) if with_res else None
    gamma = 1.0 + 0.3 * g.standard_normal(cols) if with_gamma else None
    dy = g.standard_normal((rows, cols)); dh = g.standard_normal((rows, cols))
    eps = 1e-6
    f = orc.rmsnorm_residual_fwd(x, res, gamma, eps)
    tx = torch.tensor(x, requires_grad=True)
    tr = torch.tensor(res, requires_grad=True) if with_res else None
    tg = torch.tensor(gamma, requires_grad=True) if with_gamma else None
    th, ty = _torch_rmsr(tx, tr, tg, eps)
    np.testing.assert_allclose(f["h"], th.detach().numpy(), rtol=0, atol=1e-15)
    np.testing.assert_allclose(f["y"], ty.detach().numpy(), rtol=1e-12, atol=1e-12)
    (ty * torch.tensor(dy)).sum().backward(inputs=[tx] + ([tg] if with_gamma else []),
                                           retain_graph=True)
    gx = tx.grad.numpy() + dh  # the fork's own gradient passes straight through
    b = orc.rmsnorm_residual_bwd(dy, dh, x, res, gamma, eps)
    np.testing.assert_allclose(b["dx"], gx, rtol=1e-11, atol=1e-11)
    if with_gamma:
        np.testing.assert_allclose(b["dgamma"], tg.grad.numpy(), rtol=1e-11, atol=1e-11)


def test_rmsnorm_residual_reduces_to_plain_rmsnorm(orc):
    g = _rng(51)
    x = g.standard_normal((4, 32))
    f = orc.rmsnorm_residual_fwd(x, None, None, 1e-6)
    y, rstd = orc.rmsnorm_fwd(x, 1e-6)
    np.testing.assert_array_equal(f["y"], y)
    np.testing.assert_array_equal(f["rstd"], rstd)
    dy = g.standard_normal((4, 32))
    np.testing.assert_allclose(orc.rmsnorm_residual_bwd(dy, None, x, None, None, 1e-6)["dx"],
                               orc.rmsnorm_bwd(dy, x, 1e-6), rtol=1e-14, atol=1e-14)


def test_rmsnorm_residual_dgamma_closed_form_and_fd(orc):
    """dgamma = sum_t dy * y / gamma (y = h rho gamma); and central differences."""
    g = _rng(52)
    rows, cols = 5, 12
    x = g.standard_normal((rows, cols)); res = g.standard_normal((rows, cols))
    gamma = 1.0 + 0.5 * g.random(cols); dy = g.standard_normal((rows, cols))
    f = orc.rmsnorm_residual_fwd(x, res, gamma, 1e-6)
    b = orc.rmsnorm_residual_bwd(dy, None, x, res, gamma, 1e-6)
    np.testing.assert_allclose(b["dgamma"], np.sum(dy * f["y"], axis=0) / gamma, rtol=1e-12)
    L = lambda gg: float(np.sum(dy * orc.rmsnorm_residual_fwd(x, res, gg, 1e-6)["y"]))  # noqa
    h = 1e-6
    fd = [(L(gamma + h * e) - L(gamma - h * e)) / (2 * h) for e in np.eye(cols)]
    _assert_fd(fd, b["dgamma"])


def test_rmsnorm_residual_zero_row_is_finite(orc):
    x = np.zeros((2, 8)); x[1] = np.arange(8.0)
    f = orc.rmsnorm_residual_fwd(x, None, np.ones(8), 1e-6)
    assert np.all(np.isfinite(f["y"])) and np.all(f["y"][0] == 0.0)
    b = orc.rmsnorm_residual_bwd(np.ones((2, 8)), None, x, None, np.ones(8), 1e-6)
    np.testing.assert_allclose(b["dx"][0], np.full(8, 1.0 / np.sqrt(1e-6)), rtol=1e-12)


# ----------------------------------------------------------------------------
# aggregate + weighted RMSNorm
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("n", [4, 8])
def test_aggregate_rmsnorm_matches_autograd(orc, n):
    g = _rng(60 + n)
    T, C = 4, 16
    x = g.standard_normal((T, n, C)); H = g.random((T, n)); gamma = 1.0 + 0.2 * g.standard_normal(C)
    dyn = g.standard_normal((T, C)); dy = g.standard_normal((T, C))
    eps = 1e-6
    tx = torch.tensor(x, requires_grad=True); tH = torch.tensor(H, requires_grad=True)
    tg = torch.tensor(gamma, requires_grad=True)
    ty = torch.einsum("ti,tic->tc", tH, tx)
    tyn = torch.nn.functional.rms_norm(ty, (C,), weight=tg, eps=eps)
    f = orc.h_aggregate_rmsnorm_fwd(x, H, gamma, eps)
    np.testing.assert_allclose(f["y"], ty.detach().numpy(), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(f["yn"], tyn.detach().numpy(), rtol=1e-12, atol=1e-12)
    ((tyn * torch.tensor(dyn)).sum() + (ty * torch.tensor(dy)).sum()).backward()
    b = orc.h_aggregate_rmsnorm_bwd(dyn, dy, x, H, gamma, eps)
    np.testing.assert_allclose(b["dx"], tx.grad.numpy(), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(b["dH_pre"], tH.grad.numpy(), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(b["dgamma"], tg.grad.numpy(), rtol=1e-11, atol=1e-11)


# ----------------------------------------------------------------------------
# channel-sharded proj_rms_compute_h
# ----------------------------------------------------------------------------

def _shard(x, W, C, c0, c1):
    """Channels [c0, c1) of every stream: x [T, n, C] -> [T, n, Cs]; W rows
    i*C + c -> i*Cs + (c - c0)."""
    n = x.shape[1]
    xs = np.ascontiguousarray(x[:, :, c0:c1])
    Ws = np.concatenate([W[i * C + c0:i * C + c1] for i in range(n)], axis=0)
    return xs, Ws


@pytest.mark.parametrize("n", [4, 8])
def test_partials_sum_to_numpy_matmul(orc, n):
    g = _rng(70 + n)
    T, C = 3, 24
    O = n * n + 2 * n
    x = g.standard_normal((T, n, C)); W = 0.3 * g.standard_normal((n * C, O))
    cuts = [0, 8, 16, 24]
    u = np.zeros((T, O)); s = np.zeros(T)
    for c0, c1 in zip(cuts[:-1], cuts[1:]):
        xs, Ws = _shard(x, W, C, c0, c1)
        p = orc.proj_rms_partials(xs, Ws)
        np.testing.assert_allclose(p["u"], xs.reshape(T, -1) @ Ws, rtol=1e-12, atol=1e-12)
        u += p["u"]; s += p["s"]
    np.testing.assert_allclose(u, x.reshape(T, -1) @ W, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(s, np.sum(x.reshape(T, -1) ** 2, axis=1), rtol=1e-13)


@pytest.mark.parametrize("n", [4, 8])
def test_sharded_compute_h_equals_unsharded(orc, n):
    """Totals over shards + compute_h = the (pinned) unsharded oracle, forward
    and backward; the shards' dx and dW tile the unsharded dx and dW."""
    g = _rng(80 + n)
    T, C = 3, 16
    O = n * n + 2 * n
    K = n * C
    x = g.standard_normal((T, n, C)); W = 0.3 * g.standard_normal((K, O))
    alpha = np.array([0.7, 1.1, 0.9]); b = 0.5 * g.standard_normal(O)
    iters, eps_sk, eps_rms = 20, 1e-6, 1e-6
    ref = orc.proj_rms_compute_h_fwd(x, W, alpha, b, n, iters, eps_sk, eps_rms)
    cuts = [0, 8, 16]
    shards = [_shard(x, W, C, c0, c1) for c0, c1 in zip(cuts[:-1], cuts[1:])]
    u = sum(orc.proj_rms_partials(xs, Ws)["u"] for xs, Ws in shards)
    s = sum(orc.proj_rms_partials(xs, Ws)["s"] for xs, Ws in shards)
    h = orc.compute_h_from_sums(u, s, K, alpha, b, n, iters, eps_sk, eps_rms)
    for k in ("H_pre", "H_post", "H_res"):
        np.testing.assert_allclose(h[k], ref[k], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(h["r"], ref["r"], rtol=1e-13)
    dHp = g.standard_normal((T, n)); dHq = g.standard_normal((T, n)); dHr = g.standard_normal((T, n, n))
    rb = orc.proj_rms_compute_h_bwd(dHp, dHq, dHr, x, W, alpha, b, n, iters, eps_sk, eps_rms)
    cb = orc.compute_h_bwd_from_sums(dHp, dHq, dHr, u, s, K, alpha, b, n, iters, eps_sk, eps_rms)
    np.testing.assert_allclose(cb["dalpha"], rb["dalpha"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(cb["db"], rb["db"], rtol=1e-11, atol=1e-12)
    dx = np.zeros((T, n, C)); dW = np.zeros((K, O))
    for (c0, c1), (xs, Ws) in zip(zip(cuts[:-1], cuts[1:]), shards):
        pb = orc.proj_rms_partial_bwd(xs, Ws, cb["du"], cb["coef"])
        dx[:, :, c0:c1] = pb["dx"]
        for i in range(n):
            dW[i * C + c0:i * C + c1] = pb["dW"][i * (c1 - c0):(i + 1) * (c1 - c0)]
    np.testing.assert_allclose(dx.reshape(T, -1), rb["dx"].reshape(T, -1), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dW, rb["dW"], rtol=1e-10, atol=1e-12)


def test_compute_h_bwd_du_coef_match_autograd(orc):
    """du = dL/du and coef = dL/ds * 2 (since ds/dx = 2x) from torch autograd of
    z = alpha_seg u / (sqrt(s/K) + eps) + b, the gates and the Sinkhorn."""
    from tests.test_oracle_pins import _torch_sinkhorn
    g = _rng(90)
    T, n, K = 3, 4, 32
    O = n * n + 2 * n
    u = g.standard_normal((T, O)); s = 1.0 + g.random(T) * K
    alpha = np.array([0.7, 1.1, 0.9]); b = 0.5 * g.standard_normal(O)
    iters, eps_sk, eps_rms = 20, 1e-6, 1e-6
    dHp = g.standard_normal((T, n)); dHq = g.standard_normal((T, n)); dHr = g.standard_normal((T, n, n))
    tu = torch.tensor(u, requires_grad=True); ts = torch.tensor(s, requires_grad=True)
    a = torch.tensor(np.concatenate([np.full(n, alpha[0]), np.full(n, alpha[1]),
                                     np.full(n * n, alpha[2])]))
    r = 1.0 / (torch.sqrt(ts / K) + eps_rms)
    z = a * r[:, None] * tu + torch.tensor(b)
    Hp = torch.sigmoid(z[:, :n]); Hq = 2 * torch.sigmoid(z[:, n:2 * n])
    Hr = _torch_sinkhorn(z[:, 2 * n:].reshape(T, n, n), iters, eps_sk)
    L = (Hp * torch.tensor(dHp)).sum() + (Hq * torch.tensor(dHq)).sum() + (Hr * torch.tensor(dHr)).sum()
    L.backward()
    cb = orc.compute_h_bwd_from_sums(dHp, dHq, dHr, u, s, K, alpha, b, n, iters, eps_sk, eps_rms)
    np.testing.assert_allclose(cb["du"], tu.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(cb["coef"], 2.0 * ts.grad.numpy(), rtol=1e-10, atol=1e-13)


# ----------------------------------------------------------------------------
# cross-layer fusion: post-mix of layer l -> proj_rms_compute_h of layer l+1
# ----------------------------------------------------------------------------

def test_bf16_rne_ties_and_subnormals(orc):
    """Round-to-nearest-even at 8 significant bits, from worked cases: a tie
    at 1 + 2^-8 goes down to the even 1, 1 + 3*2^-8 up to 1 + 2^-6; 255.5 and
    257 are ties that go to 256; in the subnormal range the spacing is
    2^-133, so 1.5 * 2^-133 rounds to 2^-132."""
    v = np.array([1.0, 1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8 + 2.0 ** -12), 255.5,
                  257.0, 1.5 * 2.0 ** -133, 0.0, 2.0 ** -126 * (1 + 2.0 ** -7)])
    want = np.array([1.0, 1.0, 1 + 2.0 ** -6, -(1 + 2.0 ** -7), 256.0, 256.0, 2.0 ** -132, 0.0,
                     2.0 ** -126 * (1 + 2.0 ** -7)])
    np.testing.assert_array_equal(orc.bf16_rne(v), want)


def test_bf16_rne_matches_bit_rounding(orc):
    """The arithmetic rounding agrees with the bit-level rounding of fp32
    (add 0x7FFF plus the kept lsb, truncate) on values of every magnitude."""
    import mhc_inputs as mi
    g = _rng(77)
    x = (g.standard_normal(50000) * 10.0 ** g.integers(-35, 35, 50000)).astype(np.float32)
    x = x[np.isfinite(x)]
    want = mi.bf16_bits_to_f32(mi.bf16_bits(x)).astype(np.float64)
    np.testing.assert_array_equal(orc.bf16_rne(x.astype(np.float64)), want)


def _fused_inputs(g, T, n, C):
    res = orc_bf16(g.standard_normal((T, n, C)))
    f = orc_bf16(g.standard_normal((T, C)))
    bias = orc_bf16(0.02 * g.standard_normal(C))
    W = 0.05 * g.standard_normal((n * C, n * n + 2 * n))
    alpha = np.array([0.7, 0.9, 1.1])
    b = g.standard_normal(n * n + 2 * n)
    return res, f, bias, W, alpha, b


def orc_bf16(a):
    import mhc_inputs as mi
    return mi.bf16_bits_to_f32(mi.bf16_bits(np.asarray(a, dtype=np.float32))).astype(np.float64)


@pytest.mark.parametrize("n", [4, 8])
def test_fused_next_layer_sees_permuted_residual(orc, n):
    """H_res a permutation per token and H_post = 0: layer l's output is the
    residual with its streams permuted (exact in bf16), so layer l+1's H must
    be the plain proj_rms_compute_h of that permuted tensor, and not of the
    residual itself."""
    g = _rng(90 + n)
    T, C = 6, 16
    res, f, bias, W, alpha, b = _fused_inputs(g, T, n, C)
    Hres = np.zeros((T, n, n))
    perms = [g.permutation(n) for _ in range(T)]
    for t, p in enumerate(perms):
        Hres[t, np.arange(n), p] = 1.0  # stream j goes to output stream p[j]
    Hpost = np.zeros((T, n))
    got = orc.h_post_bda_compute_h_fwd(res, f, bias, Hres, Hpost, W, alpha, b, n, 20, 1e-6, 1e-6)
    moved = np.empty_like(res)
    for t, p in enumerate(perms):
        moved[t, p] = res[t]
    np.testing.assert_array_equal(got["x_next"], moved)
    want = orc.proj_rms_compute_h_fwd(moved, W, alpha, b, n, 20, 1e-6, 1e-6)
    for k in ("H_pre", "H_post", "H_res", "u", "r"):
        np.testing.assert_array_equal(got[k], want[k])
    other = orc.proj_rms_compute_h_fwd(res, W, alpha, b, n, 20, 1e-6, 1e-6)
    assert np.max(np.abs(other["u"] - got["u"])) > 1e-3


def test_fused_next_layer_reads_rounded_output(orc):
    """Layer l+1's sum of squares is that of the bf16-rounded output, the
    tensor it would read back: r = 1/(sqrt(sum bf16(out)^2 / K) + eps), and u
    is bf16(out) . W, both checked with numpy; the unrounded output gives a
    different r."""
    g = _rng(95)
    T, n, C = 5, 4, 24
    res, f, bias, W, alpha, b = _fused_inputs(g, T, n, C)
    Hres = g.random((T, n, n))
    Hpost = 2 * g.random((T, n))
    got = orc.h_post_bda_compute_h_fwd(res, f, bias, Hres, Hpost, W, alpha, b, n, 20, 1e-6, 1e-6)
    out = np.einsum("tji,tjc->tic", Hres, res) + Hpost[:, :, None] * (f + bias)[:, None, :]
    np.testing.assert_allclose(got["out"], out, rtol=1e-13, atol=1e-13)
    xr = orc.bf16_rne(out).reshape(T, n * C)
    K = n * C
    r = 1.0 / (np.sqrt(np.sum(xr * xr, axis=1) / K) + 1e-6)
    np.testing.assert_allclose(got["r"], r, rtol=1e-13)
    np.testing.assert_allclose(got["u"], xr @ W, rtol=1e-12, atol=1e-12)
    r_exact = 1.0 / (np.sqrt(np.sum(out.reshape(T, K) ** 2, axis=1) / K) + 1e-6)
    assert np.max(np.abs(r_exact - got["r"])) > 1e-7
