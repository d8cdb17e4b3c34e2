"""Pins of the oracle's gated delta rule against things other than itself:
a hand-worked example (tests/golden), special cases with exact answers
(beta = 0, retrieval with orthonormal keys, k = 0), a brute-force evaluation
through explicit (I - beta k k^T) matrix products in reverse order, a norm
bound, the chunked (WY/UT) form against the token form, the UT transform
against a library inverse, split-and-carry against one pass, the affine
dependence on the initial state, and the slot rules of prefill / decode /
MTP / snapshot."""
import math

import numpy as np
import pytest

import oracle
from tests.golden.load import load


def _rand_chain(rng, T, dk, dv, low_decay=False):
    q = rng.normal(size=(T, dk))
    k = rng.normal(size=(T, dk))
    v = rng.normal(size=(T, dv))
    A = rng.uniform(math.log(0.001), math.log(0.01)) if low_decay else rng.uniform(0, math.log(16))
    g = -math.exp(A) * np.log1p(np.exp(rng.normal(size=T)))
    beta = 1.0 / (1.0 + np.exp(-rng.normal(size=T)))
    return q, k, v, g, beta


def _unit_rows(x, eps=oracle.L2NORM_EPS):
    return x / np.sqrt((x * x).sum(-1, keepdims=True) + eps)


# ------------------------------------------------------------ worked case ---

def test_worked_example():
    d = load("recurrence_worked.txt")
    o, S = oracle.recurrent_chain(d["q"], d["k"], d["v"], d["g"], d["beta"],
                                  scale=1.0, l2norm_qk=False)
    np.testing.assert_allclose(o, d["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(S, d["S_final"], rtol=0, atol=1e-14)


# ---------------------------------------------------------- special cases ---

def test_beta_zero_only_decays():
    rng = np.random.default_rng(1)
    T, dk, dv = 9, 5, 3
    q, k, v, g, _ = _rand_chain(rng, T, dk, dv)
    S0 = rng.normal(size=(dv, dk))
    o, S = oracle.recurrent_chain(q, k, v, g, np.zeros(T), S0=S0, scale=0.7)
    np.testing.assert_allclose(S, S0 * math.exp(g.sum()), rtol=1e-13)
    qn = _unit_rows(q)
    for t in range(T):
        St = S0 * math.exp(g[:t + 1].sum())
        np.testing.assert_allclose(o[t], 0.7 * St @ qn[t], rtol=1e-12, atol=1e-300)


def test_zero_key_only_decays():
    rng = np.random.default_rng(2)
    T, dk, dv = 6, 4, 4
    q, _, v, g, beta = _rand_chain(rng, T, dk, dv)
    S0 = rng.normal(size=(dv, dk))
    _, S = oracle.recurrent_chain(q, np.zeros((T, dk)), v, g, beta, S0=S0)
    np.testing.assert_allclose(S, S0 * math.exp(g.sum()), rtol=1e-13)


def test_orthonormal_retrieval():
    """beta = 1, g = 0, orthonormal keys, S0 = 0: writing (k_j, v_j) then
    reading with q = k_j (beta = 0 on the read tokens) returns v_j."""
    rng = np.random.default_rng(3)
    n, dv = 8, 5
    Qm, _ = np.linalg.qr(rng.normal(size=(n, n)))
    keys = Qm.T                                       # rows orthonormal
    vals = rng.normal(size=(n, dv))
    perm = rng.permutation(n)
    k = np.concatenate([keys, keys[perm]], 0)         # read tokens: key is irrelevant (beta 0)
    v = np.concatenate([vals, np.zeros((n, dv))], 0)
    q = np.concatenate([rng.normal(size=(n, n)), keys[perm]], 0)
    beta = np.concatenate([np.ones(n), np.zeros(n)])
    o, S = oracle.recurrent_chain(q, k, v, np.zeros(2 * n), beta, scale=1.0, l2norm_qk=False)
    np.testing.assert_allclose(o[n:], vals[perm], rtol=0, atol=1e-12)
    np.testing.assert_allclose(S, vals.T @ keys, rtol=0, atol=1e-12)


def _brute_force(q, k, v, g, beta, S0, scale):
    """S_T = S0 prod_t a_t (I - b_t k_t k_t^T) + sum_j b_j v_j k_j^T prod_{m>j} ...,
    products formed from the last token backwards; o_t from S_t."""
    T, dk = k.shape
    kn, qn = _unit_rows(k), _unit_rows(q)
    M = [math.exp(g[t]) * (np.eye(dk) - beta[t] * np.outer(kn[t], kn[t])) for t in range(T)]
    outs, states = [], []
    for t_end in range(1, T + 1):
        right = np.eye(dk)                              # prod_{m > j} M_m (for j = t_end-1 down)
        S = np.zeros((v.shape[1], dk))
        for j in range(t_end - 1, -1, -1):
            S += beta[j] * np.outer(v[j], kn[j]) @ right
            right = M[j] @ right
        S += S0 @ right
        states.append(S)
        outs.append(scale * S @ qn[t_end - 1])
    return np.array(outs), states[-1]


@pytest.mark.parametrize("dk,dv", [(3, 2), (2, 5), (4, 4)])
def test_brute_force_products(dk, dv):
    rng = np.random.default_rng(10 + dk * dv)
    T = 7
    q, k, v, g, beta = _rand_chain(rng, T, dk, dv, low_decay=True)
    S0 = rng.normal(size=(dv, dk))
    o, S = oracle.recurrent_chain(q, k, v, g, beta, S0=S0, scale=0.37)
    o_bf, S_bf = _brute_force(q, k, v, g, beta, S0, 0.37)
    np.testing.assert_allclose(o, o_bf, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(S, S_bf, rtol=1e-11, atol=1e-12)


def test_one_token_matrix_form():
    rng = np.random.default_rng(11)
    dk, dv = 6, 3
    q, k, v, g, beta = _rand_chain(rng, 1, dk, dv)
    S0 = rng.normal(size=(dv, dk))
    o, S = oracle.recurrent_chain(q, k, v, g, beta, S0=S0, scale=2.0)
    kn, qn = _unit_rows(k)[0], _unit_rows(q)[0]
    S1 = math.exp(g[0]) * S0 @ (np.eye(dk) - beta[0] * np.outer(kn, kn)) + beta[0] * np.outer(v[0], kn)
    np.testing.assert_allclose(S, S1, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(o[0], 2.0 * S1 @ qn, rtol=1e-13, atol=1e-14)


def test_norm_bound():
    """For beta in [0, 1] and unit k, ||I - beta k k^T||_2 <= 1, so
    ||S_t||_2 <= alpha_t ||S_{t-1}||_2 + beta_t ||v_t||."""
    rng = np.random.default_rng(12)
    T, dk, dv = 40, 8, 6
    q, k, v, g, beta = _rand_chain(rng, T, dk, dv, low_decay=True)
    S = rng.normal(size=(dv, dk))
    for t in range(T):
        _, S_new = oracle.recurrent_chain(q[t:t + 1], k[t:t + 1], v[t:t + 1], g[t:t + 1],
                                          beta[t:t + 1], S0=S)
        lhs = np.linalg.norm(S_new, 2)
        rhs = math.exp(g[t]) * np.linalg.norm(S, 2) + beta[t] * np.linalg.norm(v[t]) * \
            np.linalg.norm(_unit_rows(k[t:t + 1])[0])
        assert lhs <= rhs * (1 + 1e-12)
        S = S_new


# ------------------------------------------------------- chunked UT form ---

@pytest.mark.parametrize("T,chunk", [(64, 16), (50, 16), (1, 16), (33, 1), (70, 64), (200, 64), (16, 7)])
@pytest.mark.parametrize("low_decay", [False, True])
def test_chunked_equals_token_form(T, chunk, low_decay):
    rng = np.random.default_rng(T * 100 + chunk)
    dk, dv = 12, 9
    q, k, v, g, beta = _rand_chain(rng, T, dk, dv, low_decay)
    S0 = rng.normal(size=(dv, dk))
    o1, S1 = oracle.recurrent_chain(q, k, v, g, beta, S0=S0, scale=0.5)
    o2, S2 = oracle.chunked_chain(q, k, v, g, beta, chunk, S0=S0, scale=0.5)
    scale_o = np.abs(o1).max()
    assert np.abs(o1 - o2).max() <= 1e-10 * scale_o
    assert np.abs(S1 - S2).max() <= 1e-10 * np.abs(S1).max()


def test_ut_transform_is_inverse():
    rng = np.random.default_rng(20)
    n, dk = 16, 8
    kn = _unit_rows(rng.normal(size=(n, dk)))
    beta = rng.uniform(0, 1, n)
    gcum = np.cumsum(-rng.uniform(0, 0.2, n))
    Tm = oracle.ut_transform(kn, beta, gcum)
    A = np.zeros((n, n))
    for j in range(n):
        for m in range(j):
            A[j, m] = beta[j] * math.exp(gcum[j] - gcum[m]) * kn[j] @ kn[m]
    np.testing.assert_allclose(Tm, np.linalg.inv(np.eye(n) + A), rtol=1e-12, atol=1e-13)
    assert np.allclose(np.triu(Tm, 1), 0) and np.allclose(np.diag(Tm), 1)


# --------------------------------------------------------- pools & slots ---

def _batch(rng, lens, hqk, hv, dk, dv, low_decay=True):
    T = sum(lens)
    q = rng.normal(size=(T, hqk, dk))
    k = rng.normal(size=(T, hqk, dk))
    v = rng.normal(size=(T, hv, dv))
    A = rng.uniform(math.log(0.001), math.log(0.01), hv) if low_decay else rng.uniform(0, 2.7, hv)
    g = -np.exp(A)[None] * np.log1p(np.exp(rng.normal(size=(T, hv))))
    beta = 1.0 / (1.0 + np.exp(-rng.normal(size=(T, hv))))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    return q, k, v, g, beta, cu


def test_head_map_groups_are_contiguous():
    """V head h reads QK head h // (hv / hqk): heads 0,1 -> 0 and 2,3 -> 1."""
    rng = np.random.default_rng(30)
    q, k, v, g, beta, cu = _batch(rng, [6], 2, 4, 4, 3)
    pool = np.zeros((1, 4, 3, 4))
    o, _, _ = oracle.gdn_prefill(q, k, v, g, beta, cu, pool, [-1], [-1], 1.0)
    for h in range(4):
        oh, _ = oracle.recurrent_chain(q[:, h // 2], k[:, h // 2], v[:, h], g[:, h], beta[:, h])
        np.testing.assert_array_equal(o[:, h], oh)


@pytest.mark.parametrize("split", [1, 17, 32, 33, 63])
def test_split_and_carry_equals_one_pass(split):
    rng = np.random.default_rng(40 + split)
    T, hqk, hv, dk, dv = 64, 1, 2, 8, 6
    q, k, v, g, beta, _ = _batch(rng, [T], hqk, hv, dk, dv)
    pool = rng.normal(0, 0.5, size=(3, hv, dv, dk))
    one = np.array([0, T])
    o_full, upd_full, _ = oracle.gdn_prefill(q, k, v, g, beta, one, pool, [0], [2], 0.3)
    # first part: slot 0 -> slot 1, second part: slot 1 -> slot 1 (in place)
    sl1 = slice(0, split)
    sl2 = slice(split, T)
    o1, upd1, _ = oracle.gdn_prefill(q[sl1], k[sl1], v[sl1], g[sl1], beta[sl1], [0, split],
                                     pool, [0], [1], 0.3)
    pool1 = oracle.apply_updates(pool, upd1)
    o2, upd2, _ = oracle.gdn_prefill(q[sl2], k[sl2], v[sl2], g[sl2], beta[sl2], [0, T - split],
                                     pool1, [1], [1], 0.3, chunk=16)
    np.testing.assert_allclose(np.concatenate([o1, o2]), o_full, rtol=1e-10, atol=1e-12)
    for h in range(hv):
        np.testing.assert_allclose(upd2[(1, h)], upd_full[(2, h)], rtol=1e-10, atol=1e-12)


def test_varlen_prefill_pool_rules():
    rng = np.random.default_rng(50)
    lens = [5, 0, 19, 1]
    hqk, hv, dk, dv = 1, 2, 4, 4
    q, k, v, g, beta, cu = _batch(rng, lens, hqk, hv, dk, dv)
    pool = rng.normal(size=(6, hv, dv, dk))
    init = [2, 3, -1, 4]
    final = [2, 5, 1, -1]
    o, upd, finals = oracle.gdn_prefill(q, k, v, g, beta, cu, pool, init, final, 1.0, chunk=4)
    o_t, upd_t, _ = oracle.gdn_prefill(q, k, v, g, beta, cu, pool, init, final, 1.0)
    np.testing.assert_allclose(o, o_t, rtol=1e-10, atol=1e-12)
    assert set(upd) == {(2, 0), (2, 1), (5, 0), (5, 1), (1, 0), (1, 1)}
    for h in range(hv):
        np.testing.assert_array_equal(upd[(5, h)], pool[3, h])        # empty sequence: copy
        np.testing.assert_allclose(upd[(2, h)], upd_t[(2, h)], rtol=1e-10, atol=1e-12)
        _, S = oracle.recurrent_chain(q[5:24, 0], k[5:24, 0], v[5:24, h], g[5:24, h], beta[5:24, h])
        np.testing.assert_allclose(upd[(1, h)], S, rtol=1e-10, atol=1e-12)   # zero init


def test_decode_and_mtp_slot_rules():
    """decode in place == prefill of the same tokens; MTP snapshots hold the
    state after each token and leave the source slot alone; a negative slot
    gives zero output; snapshot copy moves whole slots."""
    rng = np.random.default_rng(60)
    N, tps, hqk, hv, dk, dv = 3, 4, 1, 2, 4, 3
    q, k, v, g, beta, _ = _batch(rng, [N * tps], hqk, hv, dk, dv)
    pool = rng.normal(size=(20, hv, dv, dk))
    idx = np.array([7, -1, 2])
    o_d, upd_d = oracle.gdn_decode(q, k, v, g, beta, tps, pool, idx, scale=0.5)
    cu = np.arange(N + 1) * tps
    o_p, upd_p, _ = oracle.gdn_prefill(q, k, v, g, beta, cu, pool, idx, idx, 0.5)
    live = np.r_[0:tps, 2 * tps:3 * tps]
    np.testing.assert_array_equal(o_d[live], o_p[live])
    assert upd_d.keys() == upd_p.keys()
    assert np.all(o_d[tps:2 * tps] == 0)          # padding row: zero output (prefill would run it)

    snap = np.array([[10, 11, 12, 13], [14, 15, 16, 17], [18, -1, 19, 0]])
    o_s, upd_s = oracle.gdn_decode(q, k, v, g, beta, tps, pool, idx, snap, scale=0.5)
    np.testing.assert_array_equal(o_s, o_d)
    assert (7, 0) not in upd_s and (2, 1) not in upd_s
    for i in (0, 2):
        for t in range(tps):
            if snap[i, t] < 0:
                continue
            r = slice(i * tps, i * tps + t + 1)
            for h in range(hv):
                _, S = oracle.recurrent_chain(q[r, 0], k[r, 0], v[r, h], g[r, h], beta[r, h],
                                              S0=pool[idx[i], h], scale=0.5)
                np.testing.assert_array_equal(upd_s[(snap[i, t], h)], S)
    cp = oracle.state_snapshot(pool, [3, -1, 5], [5, 1, 3])
    assert set(cp) == {5, 3}
    np.testing.assert_array_equal(cp[5], pool[3])
    np.testing.assert_array_equal(cp[3], pool[5])          # swap: reads see the old pool


def test_layer_chunked_equals_token_tiny():
    import workloads
    w = workloads.tiny()
    d = w.dims
    res = {}
    for ch in (None, w.chunk):
        res[ch] = oracle.layer_prefill(w.x, w.cu_seqlens, w.conv_w, None, w.conv_pool, w.A_log,
                                       w.dt_bias, w.a, w.b, w.state_pool, w.slots,
                                       w.has_initial_state, d.hqk, d.hv, d.dk, d.dv, w.scale,
                                       chunk=ch)
    o1, o2 = res[None][0], res[w.chunk][0]
    assert np.abs(o1 - o2).max() <= 1e-10 * np.abs(o1).max()
    for key in res[None][2]:
        np.testing.assert_allclose(res[w.chunk][2][key], res[None][2][key], rtol=1e-9, atol=1e-12)


# ------------------------------------------------- affine state map (scan) --

@pytest.mark.parametrize("form", ["token", "chunked"])
def test_state_map_is_affine_in_the_initial_state(form):
    """The chain is affine in its initial state: with dv = dk the identity is
    a state, the transition is A = S_end(I) - S_end(0), and for any S0,
    S_end(S0) = S0 A + S_end(0) and o_t(S0) - o_t(0) = S0 (o_t(I) - o_t(0)).
    Composing two segments' affine maps equals one pass over both.  These
    are the identities a chunk-state scan over one long sequence rests on."""
    rng = np.random.default_rng(71 if form == "token" else 72)
    d, T, m = 16, 53, 20
    q, k, v, g, beta = _rand_chain(rng, T, d, d)

    def run(S0, lo=0, hi=T):
        args = (q[lo:hi], k[lo:hi], v[lo:hi], g[lo:hi], beta[lo:hi])
        if form == "token":
            return oracle.recurrent_chain(*args, S0=S0, scale=0.3)
        return oracle.chunked_chain(*args, chunk=8, S0=S0, scale=0.3)

    o0, B = run(np.zeros((d, d)))
    oI, MI = run(np.eye(d))
    A = MI - B
    S0 = rng.normal(size=(d, d)) * 0.1
    oS, SS = run(S0)
    np.testing.assert_allclose(SS, S0 @ A + B, rtol=0, atol=1e-10)
    np.testing.assert_allclose(oS - o0, (S0 @ (oI - o0).T).T, rtol=0, atol=1e-10)
    # two segments: [0, m) then [m, T), each as (A_p, B_p), composed
    _, B1 = run(np.zeros((d, d)), 0, m)
    _, M1 = run(np.eye(d), 0, m)
    _, B2 = run(np.zeros((d, d)), m, T)
    _, M2 = run(np.eye(d), m, T)
    composed = (S0 @ (M1 - B1) + B1) @ (M2 - B2) + B2
    np.testing.assert_allclose(composed, SS, rtol=0, atol=1e-10)
