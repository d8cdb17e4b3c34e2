"""Pins of the oracle's gating and conv1d against things other than itself:
hand-derived worked values (tests/golden), PyTorch's fp64 library routines
(softplus, sigmoid, conv1d, silu), and the token-by-token == whole-sequence
consistency of the conv update."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from tests.golden.load import load


# ---------------------------------------------------------------- gating ----

def test_gating_worked_values():
    d = load("gating_worked.txt")
    hv = len(d["A_log"])
    # one token per head: put row r on head r
    a = d["a"].reshape(1, hv)
    b = d["b"].reshape(1, hv)
    g, beta = oracle.gating(a, b, d["A_log"], d["dt_bias"])
    np.testing.assert_allclose(g[0], d["g"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(beta[0], d["beta"], rtol=1e-14, atol=1e-15)


def test_gating_vs_library_routines():
    rng = np.random.default_rng(0)
    T, hv = 257, 7
    a = rng.normal(0, 3, (T, hv))
    b = rng.normal(0, 3, (T, hv))
    A_log = rng.uniform(0, math.log(16), hv)
    dt_bias = rng.normal(0, 0.1, hv)
    g, beta = oracle.gating(a, b, A_log, dt_bias)
    ta = torch.from_numpy(a) + torch.from_numpy(dt_bias)
    g_ref = -torch.exp(torch.from_numpy(A_log)) * F.softplus(ta, beta=1.0, threshold=1e9)
    beta_ref = torch.sigmoid(torch.from_numpy(b))
    np.testing.assert_allclose(g, g_ref.numpy(), rtol=1e-13, atol=1e-300)
    np.testing.assert_allclose(beta, beta_ref.numpy(), rtol=1e-13, atol=1e-300)
    assert np.all(g < 0) and np.all((beta >= 0) & (beta <= 1))


def test_gating_extremes_closed_form():
    """Far from 0, softplus(x) -> x (x >> 0) or e^x (x << 0) and sigmoid -> 1
    or e^x: the oracle must reach these limits without overflow."""
    xs = np.array([[800.0, 60.0, -60.0, -800.0]])
    zero = np.zeros(4)
    g, beta = oracle.gating(xs, xs, zero, zero)
    assert np.all(np.isfinite(g)) and np.all(np.isfinite(beta))
    np.testing.assert_allclose(g[0, :2], -xs[0, :2], rtol=1e-15)
    np.testing.assert_allclose(g[0, 2], -math.exp(-60.0), rtol=1e-14)
    assert g[0, 3] == 0.0
    np.testing.assert_allclose(beta[0], [1.0, 1.0, math.exp(-60.0), 0.0], rtol=1e-14, atol=0)


def test_gating_head_broadcast():
    # A_log / dt_bias are per head: permuting heads permutes the outputs
    rng = np.random.default_rng(1)
    a, b = rng.normal(size=(5, 4)), rng.normal(size=(5, 4))
    A_log, dt = rng.uniform(0, 2, 4), rng.normal(0, 0.1, 4)
    p = [2, 0, 3, 1]
    g1, b1 = oracle.gating(a, b, A_log, dt)
    g2, b2 = oracle.gating(a[:, p], b[:, p], A_log[p], dt[p])
    np.testing.assert_array_equal(g1[:, p], g2)
    np.testing.assert_array_equal(b1[:, p], b2)


# ------------------------------------------------------------------ conv ----

def test_conv_worked_example():
    d = load("conv_worked.txt")
    y, st = oracle.conv1d_seq(d["x"], d["weight"], None, d["hist"], silu=False)
    np.testing.assert_array_equal(y, d["y"])
    np.testing.assert_array_equal(st, d["state"])
    _, st2 = oracle.conv1d_seq(d["x_short"], d["weight"], None, d["hist"], silu=False)
    np.testing.assert_array_equal(st2, d["state_short"])


def _conv_library(x, w, bias, hist, silu):
    """torch.nn.functional.conv1d (cross-correlation) on hist ++ x, fp64."""
    T, C = x.shape
    W = w.shape[1]
    ext = np.concatenate([hist if hist is not None else np.zeros((W - 1, C)), x], 0)
    if T == 0:
        return np.zeros((0, C)), ext[-(W - 1):]
    inp = torch.from_numpy(ext.T.copy()).unsqueeze(0)               # [1, C, T+W-1]
    out = F.conv1d(inp, torch.from_numpy(w).unsqueeze(1), None if bias is None else
                   torch.from_numpy(bias), groups=C)                  # valid: [1, C, T]
    if silu:
        out = F.silu(out)
    return out[0].T.numpy(), ext[-(W - 1):]


@pytest.mark.parametrize("T", [0, 1, 2, 3, 4, 37])
@pytest.mark.parametrize("with_hist", [False, True])
@pytest.mark.parametrize("with_bias", [False, True])
def test_conv_vs_torch_conv1d(T, with_hist, with_bias):
    rng = np.random.default_rng(T * 4 + with_hist * 2 + with_bias)
    C, W = 24, 4
    x = rng.normal(size=(T, C))
    w = rng.uniform(-0.5, 0.5, (C, W))
    bias = rng.normal(size=C) if with_bias else None
    hist = rng.normal(size=(W - 1, C)) if with_hist else None
    y, st = oracle.conv1d_seq(x, w, bias, hist, silu=True)
    y_ref, st_ref = _conv_library(x, w, bias, hist, True)
    np.testing.assert_allclose(y, y_ref, rtol=1e-13, atol=1e-14)
    np.testing.assert_array_equal(st, st_ref)


def test_conv_other_widths():
    rng = np.random.default_rng(5)
    for W in (2, 3, 5):
        x = rng.normal(size=(9, 6))
        w = rng.normal(size=(6, W))
        hist = rng.normal(size=(W - 1, 6))
        y, st = oracle.conv1d_seq(x, w, None, hist, silu=False)
        y_ref, st_ref = _conv_library(x, w, None, hist, False)
        np.testing.assert_allclose(y, y_ref, rtol=1e-13, atol=1e-14)
        np.testing.assert_array_equal(st, st_ref)


def test_conv_varlen_and_update_consistency():
    """Packed varlen conv == per-sequence conv; the decode update applied
    token by token == the prefill conv over those tokens; MTP snapshots hold
    the state after each token; slot < 0 gives zero rows and no write."""
    rng = np.random.default_rng(7)
    C, W, slots = 16, 4, 6
    lens = [5, 0, 1, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    x = rng.normal(size=(cu[-1], C))
    w = rng.uniform(-0.5, 0.5, (C, W))
    pool = rng.normal(size=(slots, W - 1, C))
    idx = np.array([3, 1, -1, 0])
    has = np.array([1, 1, 1, 0])
    y, upd = oracle.conv1d_fwd(x, cu, w, None, pool, idx, has)
    assert set(upd) == {3, 1, 0}
    for i in range(4):
        s, e = cu[i], cu[i + 1]
        hist = pool[idx[i]] if idx[i] >= 0 and has[i] else None
        yr, sr = _conv_library(x[s:e], w, None, hist, True)
        np.testing.assert_allclose(y[s:e], yr, rtol=1e-13, atol=1e-14)
        if idx[i] >= 0:
            np.testing.assert_array_equal(upd[idx[i]], sr)
    np.testing.assert_array_equal(upd[1], pool[1])   # empty sequence keeps its state

    # decode update, 3 tokens per sequence, in place vs snapshots
    N, tps = 2, 3
    xu = rng.normal(size=(N * tps, C))
    sidx = np.array([2, 4])
    yu, upd_u = oracle.conv1d_update(xu, tps, w, None, pool, sidx)
    snap = np.array([[0, -1, 1], [3, 5, -1]])
    ys, upd_s = oracle.conv1d_update(xu, tps, w, None, pool, sidx, snap)
    np.testing.assert_array_equal(yu, ys)
    for i in range(N):
        rows = slice(i * tps, (i + 1) * tps)
        yr, sr = _conv_library(xu[rows], w, None, pool[sidx[i]], True)
        np.testing.assert_allclose(yu[rows], yr, rtol=1e-13, atol=1e-14)
        np.testing.assert_array_equal(upd_u[sidx[i]], sr)
        for t in range(tps):
            if snap[i, t] >= 0:
                _, st = _conv_library(xu[i * tps:i * tps + t + 1], w, None, pool[sidx[i]], True)
                np.testing.assert_array_equal(upd_s[snap[i, t]], st)
    assert set(upd_s) == {0, 1, 3, 5}          # source slots 2, 4 untouched
    yp, upd_p = oracle.conv1d_update(xu, tps, w, None, pool, np.array([-1, 4]))
    assert np.all(yp[:tps] == 0) and set(upd_p) == {4}
