"""Pins of the fp32 pinned-order reference (oracle/mhc_oracle_pinned.c), the
reference of the library's bit-reproducible mode.

The contract (RL-Align/RL-Kernel PR #383, PR body, "Numerical contract"):
fp32 arithmetic, the four-stream tree (a0 + a1) + (a2 + a3) and a serial
ascending left fold for long reductions.  Pinned against: hand-worked values
where the tree, the serial fold, a reordered sum and the exact sum all give
different answers (tests/golden/pinned_trees.txt); the fp64 oracle within
fp32 rounding on seeded inputs; the exp accuracy against math.exp; the
Sinkhorn row and column sums."""
import math
import os

import numpy as np
import pytest

import mhc_inputs as mi

ITERS, EPS_SK, EPS_RMS = mi.ITERS, mi.EPS_SK, mi.EPS_RMS
GOLD = os.path.join(os.path.dirname(__file__), "golden", "pinned_trees.txt")
E24 = float(2 ** 24)


def _golden():
    vals = {}
    with open(GOLD) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                case, key, v = line.split()
                vals[(case, key)] = float(v)
    return vals


def test_exp_accuracy(orc):
    x = np.linspace(-87.0, 88.0, 100001).astype(np.float32)
    e = orc.pin_exp(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    assert float(np.max(np.abs(e - ref) / ref)) <= 2.5 * 2.0 ** -24   # within 2.5 ulp
    assert orc.pin_exp(np.float32([0.0]))[0] == 1.0
    assert abs(float(orc.pin_exp(np.float32([1.0]))[0]) - math.e) <= 2 * 2.0 ** -23 * math.e


def test_hand_worked_trees(orc):
    g = _golden()
    adv = np.array([E24, 1.0, 1.0, -E24], np.float32)
    # aggregate: x [1, 4, 1], H_pre ones
    x = adv.reshape(1, 4, 1)
    y = orc.pin_h_aggregate_fwd(x, np.ones((1, 4), np.float32))
    assert y[0, 0] == g[("agg_tree", "y")]
    # aggregate backward: stream 0 over 4 channels
    xb = np.zeros((1, 4, 4), np.float32)
    xb[0, 0] = adv
    _, dH = orc.pin_h_aggregate_bwd(np.ones((1, 4), np.float32), xb, np.ones((1, 4), np.float32))
    assert dH[0, 0] == g[("agg_fold", "dH_pre0")]
    # post-mix: H_res column 0 all ones
    Hr = np.zeros((1, 4, 4), np.float32)
    Hr[0, :, 0] = 1.0
    out = orc.pin_h_post_bda_fwd(x, np.zeros((1, 1), np.float32), np.zeros(1, np.float32), Hr,
                                 np.zeros((1, 4), np.float32))
    assert out[0, 0, 0] == g[("post_tree", "out0")] and np.all(out[0, 1:, 0] == 0)
    # the same inputs under the other orders give other answers (the pins can tell)
    serial = np.float32(np.float32(np.float32(adv[0] + adv[1]) + adv[2]) + adv[3])
    assert serial == 0.0 and float(np.sum(adv.astype(np.float64))) == 2.0


def _close(a, b, rel, atol=0.0):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    assert np.all(np.abs(a - b) <= rel * np.max(np.abs(b)) + atol), float(np.max(np.abs(a - b)))


@pytest.mark.parametrize("T,C,seed,stress", [(7, 64, 1, False), (5, 40, 2, True)])
def test_pinned_matches_fp64_oracle(orc, T, C, seed, stress):
    """Every output within fp32 rounding (bf16 outputs within one bf16 ulp) of
    the fp64 definitions."""
    kw = dict(w_std=0.05, alpha=1.0, b_std=1.0) if stress else {}
    inp = mi.layer_inputs(T, 4, C, seed, **kw)
    pf = orc.pin_layer_fwd(inp, ITERS, EPS_SK, EPS_RMS)
    rf = orc.layer_fwd(inp, 4, ITERS, EPS_SK, EPS_RMS)
    for k in ("H_pre", "H_post", "H_res"):
        _close(pf[k], rf[k], 0, 2e-6)
    _close(pf["u"], rf["u"], 1e-5)
    _close(pf["r"], rf["r"], 1e-6)
    for k in ("y", "out"):
        _close(pf[k], rf[k], 0, 1e-2)
    pb = orc.pin_layer_bwd(inp, pf, ITERS, EPS_SK, EPS_RMS)
    rb = orc.layer_bwd(inp, rf, 4, ITERS, EPS_SK, EPS_RMS)
    for k in ("dx", "df"):
        r = np.asarray(rb[k], np.float64)
        assert np.all(np.abs(pb[k] - r) <= 2 ** -7 * np.abs(r) + 1e-4), k
    for k in ("dW", "dalpha", "db", "dbias"):
        _close(pb[k], rb[k], 1e-5, 1e-6)
    # the standalone ops agree with the layer composition
    s = orc.pin_proj_rms_compute_h_fwd(inp["x"], inp["W"], inp["alpha"], inp["b"], ITERS, EPS_SK,
                                       EPS_RMS)
    for k in ("H_pre", "H_post", "H_res", "u", "r"):
        assert np.array_equal(s[k], pf[k]), k


def test_pinned_sinkhorn(orc):
    inp = mi.sinkhorn_inputs(64, 4, seed=3)
    P = orc.pin_sinkhorn_fwd(inp["logits"], ITERS, EPS_SK)
    assert np.all(P >= 0)
    cs = P.sum(axis=1, dtype=np.float64)   # columns after the last (column) step
    assert np.all(np.abs(cs - (1 - EPS_SK)) <= 1e-6)
    _close(P, orc.sinkhorn_fwd(inp["logits"], ITERS, EPS_SK), 0, 2e-6)
    dl = orc.pin_sinkhorn_bwd(inp["dP"], inp["logits"], ITERS, EPS_SK)
    _close(dl, orc.sinkhorn_bwd(inp["dP"], inp["logits"], ITERS, EPS_SK), 1e-4, 1e-5)
