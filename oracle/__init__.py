"""CPU oracle for the Gated DeltaNet layer — TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library's own path never calls it
and shares no code with it: the arithmetic lives in ``gdn_oracle.c`` (plain
fp64 C, one chain at a time); this module only gathers the per-sequence,
per-head chains out of packed batches and state pools, and applies the slot
rules, in numpy.

Slot rules (the state pool is the "MambaCacheManager" buffer of the Qwen3next
pull request, Highlights; the copy between slots is the buffer copy from
source to destination indices shown in its review):
  * a slot index < 0 means "no slot": zero initial state, nothing written,
    and (decode) the output rows of that sequence are zero;
  * every read sees the pool as it was before the call;
  * decode without snapshots updates its slot in place; with snapshots the
    source slot is only read, and the state after token t goes to snap[i][t].

Pins that tie this oracle to something other than itself live in
``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_gdn.so")

L2NORM_EPS = 1e-6

_lib = None


def build_oracle(force: bool = False) -> str:
    """Compile gdn_oracle.c with the host C compiler (no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c99",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build_oracle()
        L = ctypes.CDLL(_LIB_PATH)
        P = ctypes.POINTER(ctypes.c_double)
        L.oracle_gating.argtypes = [P, P, P, P, ctypes.c_long, ctypes.c_int, P, P]
        L.oracle_conv1d_seq.argtypes = [P, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                        P, P, P, ctypes.c_int, P, P]
        L.oracle_l2norm.argtypes = [P, ctypes.c_long, ctypes.c_int, ctypes.c_double, P]
        L.oracle_gated_rmsnorm.argtypes = [P, P, P, ctypes.c_long, ctypes.c_int,
                                           ctypes.c_double, P]
        L.oracle_gdn_recurrent.argtypes = [P, P, P, P, P, ctypes.c_long, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                           ctypes.c_double, P, P, P]
        L.oracle_ut_transform.argtypes = [P, P, P, ctypes.c_int, ctypes.c_int, P]
        L.oracle_gdn_chunked.argtypes = [P, P, P, P, P, ctypes.c_long, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                         ctypes.c_double, ctypes.c_int, P, P]
        for f in (L.oracle_gating, L.oracle_conv1d_seq, L.oracle_l2norm,
                  L.oracle_gated_rmsnorm, L.oracle_gdn_recurrent, L.oracle_ut_transform,
                  L.oracle_gdn_chunked):
            f.restype = None
        _lib = L
    return _lib


def _f64(x) -> np.ndarray:
    """Contiguous float64 copy of a numpy array or a (CPU) torch tensor."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").numpy()
    return np.asarray(x, dtype=np.int64)


def _p(a: np.ndarray | None):
    if a is None:
        return ctypes.POINTER(ctypes.c_double)()
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _workers(threads: int | None) -> int:
    return max(1, threads if threads else (os.cpu_count() or 1))


# ----------------------------------------------------------------------------
# single-chain primitives (thin wrappers over the C definitions)
# ----------------------------------------------------------------------------

def gating(a, b, A_log, dt_bias):
    """g = -exp(A_log)*softplus(a + dt_bias), beta = sigmoid(b); a, b: [T, hv]."""
    a, b, A_log, dt_bias = _f64(a), _f64(b), _f64(A_log), _f64(dt_bias)
    T, hv = a.shape
    g = np.empty_like(a)
    beta = np.empty_like(a)
    lib().oracle_gating(_p(a), _p(b), _p(A_log), _p(dt_bias), T, hv, _p(g), _p(beta))
    return g, beta


def conv1d_seq(x, weight, bias=None, hist=None, silu=True):
    """One sequence: x [T, C], weight [C, W] -> (y [T, C], final state [W-1, C])."""
    x, weight = _f64(x), _f64(weight)
    T, C = x.shape
    W = weight.shape[1]
    bias = None if bias is None else _f64(bias)
    hist = None if hist is None else _f64(hist)
    y = np.empty((T, C))
    st = np.empty((W - 1, C))
    lib().oracle_conv1d_seq(_p(x), T, C, W, _p(weight), _p(bias), _p(hist), int(silu),
                            _p(y), _p(st))
    return y, st


def l2norm(x, eps=L2NORM_EPS):
    x = _f64(x)
    d = x.shape[-1]
    flat = x.reshape(-1, d)
    out = np.empty_like(flat)
    lib().oracle_l2norm(_p(flat), flat.shape[0], d, eps, _p(out))
    return out.reshape(x.shape)


RMSNORM_EPS = 1e-6


def gated_rmsnorm(o, z, weight, eps=RMSNORM_EPS):
    """y = o / sqrt(mean(o^2) + eps) * weight * SiLU(z) over the last axis."""
    o, z, w = _f64(o), _f64(z), _f64(weight)
    d = o.shape[-1]
    assert z.shape == o.shape and w.shape == (d,)
    fo, fz = o.reshape(-1, d), z.reshape(-1, d)
    y = np.empty_like(fo)
    lib().oracle_gated_rmsnorm(_p(fo), _p(fz), _p(w), fo.shape[0], d, eps, _p(y))
    return y.reshape(o.shape)


def recurrent_chain(q, k, v, g, beta, S0=None, scale=1.0, l2norm_qk=True,
                    eps=L2NORM_EPS, snapshots=False):
    """Token form for one chain. q, k [T, dk]; v [T, dv]; g, beta [T].

    Returns (o [T, dv], S_final [dv, dk]) and, if snapshots, the state after
    every token [T, dv, dk].
    """
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk)) if S0 is None else _f64(S0).copy()
    o = np.empty((T, dv))
    sn = np.empty((T, dv, dk)) if snapshots else None
    lib().oracle_gdn_recurrent(_p(q), _p(k), _p(v), _p(g), _p(beta), T, dk, dv,
                               float(scale), int(l2norm_qk), float(eps), _p(S), _p(o), _p(sn))
    return (o, S, sn) if snapshots else (o, S)


def chunked_chain(q, k, v, g, beta, chunk, S0=None, scale=1.0, l2norm_qk=True,
                  eps=L2NORM_EPS):
    """Chunked (WY/UT) form for one chain; same contract as recurrent_chain."""
    q, k, v, g, beta = _f64(q), _f64(k), _f64(v), _f64(g), _f64(beta)
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk)) if S0 is None else _f64(S0).copy()
    o = np.empty((T, dv))
    lib().oracle_gdn_chunked(_p(q), _p(k), _p(v), _p(g), _p(beta), T, dk, dv,
                             float(scale), int(l2norm_qk), float(eps), int(chunk), _p(S), _p(o))
    return o, S


def ut_transform(kn, beta, gcum):
    """(I + A)^-1 of one chunk; kn [n, dk] normalised keys, beta/gcum [n]."""
    kn, beta, gcum = _f64(kn), _f64(beta), _f64(gcum)
    n, dk = kn.shape
    Tm = np.empty((n, n))
    lib().oracle_ut_transform(_p(kn), _p(beta), _p(gcum), n, dk, _p(Tm))
    return Tm


# ----------------------------------------------------------------------------
# batch / pool level.  Pools are never copied whole (they can hold GiBs):
# each function returns the slots it writes as {slot: array} or
# {(slot, head): array}; apply_updates() folds them into a small pool.
# ----------------------------------------------------------------------------

def apply_updates(pool, updates):
    """Return a float64 copy of pool with the given slot updates written."""
    out = _f64(pool).copy()
    for key, val in updates.items():
        out[key] = val
    return out


def conv1d_fwd(x, cu_seqlens, weight, bias, conv_pool, state_indices,
               has_initial_state=None, silu=True):
    """Varlen causal conv over packed sequences.

    x [T, C]; weight [C, W]; conv_pool [slots, W-1, C]; state_indices [N].
    Returns (y [T, C], {slot: final state [W-1, C]}).  A sequence with slot
    < 0 starts from zero history and writes no state; has_initial_state[i]
    == 0 starts from zero history but still writes its final state.
    """
    x = _f64(x)
    cu = _i64(cu_seqlens)
    idx = _i64(state_indices)
    y = np.zeros_like(x)
    upd = {}
    for i in range(len(cu) - 1):
        s, e = int(cu[i]), int(cu[i + 1])
        slot = int(idx[i])
        use_hist = slot >= 0 and (has_initial_state is None or int(has_initial_state[i]) != 0)
        hist = _f64(conv_pool[slot]) if use_hist else None
        yi, st = conv1d_seq(x[s:e], weight, bias, hist, silu)
        y[s:e] = yi
        if slot >= 0:
            upd[slot] = st
    return y, upd


def conv1d_update(x, tokens_per_seq, weight, bias, conv_pool, state_indices,
                  snap_indices=None, silu=True):
    """Decode/MTP conv update; x [N*tps, C], row i*tps + t.

    Without snapshots the slot is updated in place; with snap_indices [N, tps]
    the source slot is only read and the state after token t goes to
    snap[i][t] (entries < 0 are skipped).  Rows of a sequence whose slot is
    < 0 are zero.  Returns (y, {slot: state}).
    """
    x = _f64(x)
    idx = _i64(state_indices)
    snap = None if snap_indices is None else _i64(snap_indices)
    y = np.zeros_like(x)
    upd = {}
    for i in range(len(idx)):
        slot = int(idx[i])
        if slot < 0:
            continue
        hist = _f64(conv_pool[slot])
        for t in range(tokens_per_seq):
            r = i * tokens_per_seq + t
            yi, hist = conv1d_seq(x[r:r + 1], weight, bias, hist, silu)
            y[r] = yi[0]
            if snap is not None and snap[i, t] >= 0:
                upd[int(snap[i, t])] = hist
        if snap is None:
            upd[slot] = hist
    return y, upd


def _chains(jobs, fn, threads):
    if _workers(threads) == 1 or len(jobs) <= 1:
        return [fn(j) for j in jobs]
    with ThreadPoolExecutor(max_workers=_workers(threads)) as ex:
        return list(ex.map(fn, jobs))


def gdn_prefill(q, k, v, g, beta, cu_seqlens, state_pool, init_idx, final_idx,
                scale, l2norm_qk=True, chunk=None, chains=None, threads=None):
    """Varlen prefill over packed sequences.

    q, k [T, hqk, dk]; v [T, hv, dv]; g, beta [T, hv]; state_pool
    [slots, hv, dv, dk] (read only at the initial slots).  V head h reads QK
    head h // (hv // hqk).  chunk=None runs the token form, else the chunked
    form.  chains restricts the work to a list of (seq, head) pairs.
    Returns (o [T, hv, dv] (zero outside the chains run),
             {(final slot, head): S_final}, {(seq, head): S_final}).
    """
    cu = _i64(cu_seqlens)
    ii, fi = _i64(init_idx), _i64(final_idx)
    hqk, hv, dv = q.shape[1], v.shape[1], v.shape[2]
    grp = hv // hqk
    n = len(cu) - 1
    todo = [(i, h) for i in range(n) for h in range(hv)] if chains is None else list(chains)

    def run(job):
        i, h = job
        s, e = int(cu[i]), int(cu[i + 1])
        S0 = _f64(state_pool[int(ii[i]), h]) if ii[i] >= 0 else None
        args = (q[s:e, h // grp], k[s:e, h // grp], v[s:e, h], g[s:e, h], beta[s:e, h])
        if chunk is None:
            return recurrent_chain(*args, S0=S0, scale=scale, l2norm_qk=l2norm_qk)
        return chunked_chain(*args, chunk=chunk, S0=S0, scale=scale, l2norm_qk=l2norm_qk)

    res = _chains(todo, run, threads)
    o = np.zeros((q.shape[0], hv, dv))
    upd, finals = {}, {}
    for (i, h), (oi, S) in zip(todo, res):
        s, e = int(cu[i]), int(cu[i + 1])
        o[s:e, h] = oi
        finals[(i, h)] = S
        if fi[i] >= 0:
            upd[(int(fi[i]), h)] = S
    return o, upd, finals


def gdn_decode(q, k, v, g, beta, tokens_per_seq, state_pool, state_indices,
               snap_indices=None, scale=1.0, l2norm_qk=True, seqs=None, threads=None):
    """Recurrent decode / MTP decode over a slot pool.

    q, k [N*tps, hqk, dk]; v [N*tps, hv, dv]; g, beta [N*tps, hv]; row
    i*tps + t is token t of sequence i.  Without snapshots slot idx[i] is
    updated in place; with snap_indices [N, tps] it is only read and the
    state after token t is written to snap[i][t].  seqs restricts the work
    to a subset of sequences.  Returns (o [N*tps, hv, dv],
    {(slot, head): state}).
    """
    idx = _i64(state_indices)
    snap = None if snap_indices is None else _i64(snap_indices)
    hqk, hv, dv = q.shape[1], v.shape[1], v.shape[2]
    grp = hv // hqk
    tps = tokens_per_seq
    seq_list = range(len(idx)) if seqs is None else seqs
    todo = [(i, h) for i in seq_list if idx[i] >= 0 for h in range(hv)]

    def run(job):
        i, h = job
        r0, r1 = i * tps, (i + 1) * tps
        return recurrent_chain(q[r0:r1, h // grp], k[r0:r1, h // grp], v[r0:r1, h],
                               g[r0:r1, h], beta[r0:r1, h], S0=_f64(state_pool[int(idx[i]), h]),
                               scale=scale, l2norm_qk=l2norm_qk, snapshots=True)

    res = _chains(todo, run, threads)
    o = np.zeros((q.shape[0], hv, dv))
    upd = {}
    for (i, h), (oi, S, sn) in zip(todo, res):
        o[i * tps:(i + 1) * tps, h] = oi
        if snap is None:
            upd[(int(idx[i]), h)] = S
        else:
            for t in range(tps):
                if snap[i, t] >= 0:
                    upd[(int(snap[i, t]), h)] = sn[t]
    return o, upd


def state_snapshot(pool, src, dst):
    """pool[dst[i]] <- pool[src[i]]; reads see the pool before the call.

    Returns {dst slot: copied state} (no arithmetic: a byte copy)."""
    upd = {}
    for s, d in zip(_i64(src), _i64(dst)):
        if s >= 0 and d >= 0:
            upd[int(d)] = np.array(pool[int(s)], copy=True)
    return upd


def split_qkv(y, hqk, hv, dk, dv):
    """Split the conv output [T, 2*hqk*dk + hv*dv] into q, k, v heads
    (channel order q | k | v, head-major inside each)."""
    T = y.shape[0]
    nq = hqk * dk
    q = y[:, :nq].reshape(T, hqk, dk)
    k = y[:, nq:2 * nq].reshape(T, hqk, dk)
    v = y[:, 2 * nq:2 * nq + hv * dv].reshape(T, hv, dv)
    return q, k, v


def layer_prefill(x, cu_seqlens, conv_weight, conv_bias, conv_pool, A_log, dt_bias,
                  a, b, state_pool, slots, has_initial_state, hqk, hv, dk, dv, scale,
                  chunk=None, threads=None):
    """conv1d (+SiLU) -> split -> gating -> gated delta rule for one prefill
    batch.  A sequence's conv state and recurrent state share its slot; with
    has_initial_state[i] == 0 both start from zero.

    Returns (o, {slot: conv state}, {(slot, head): S}, g, beta, y).
    """
    slots = _i64(slots)
    has = _i64(has_initial_state)
    y, conv_upd = conv1d_fwd(x, cu_seqlens, conv_weight, conv_bias, conv_pool, slots,
                             has_initial_state=has)
    q, k, v = split_qkv(y, hqk, hv, dk, dv)
    g, beta = gating(a, b, A_log, dt_bias)
    init = np.where(has != 0, slots, -1)
    o, upd, _ = gdn_prefill(q, k, v, g, beta, cu_seqlens, state_pool, init, slots,
                            scale, True, chunk, threads=threads)
    return o, conv_upd, upd, g, beta, y
