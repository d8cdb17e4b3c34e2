"""GPU parity of recurrent decode and MTP decode (with state snapshots and
accept/rollback copies) through the C ABI, against the CPU oracle, at the
full decode (256 x 1) and MTP (128 x 4) sizes and at small odd shapes."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_common import DEV, cuda, gdn, oracle_gating, qkv_views, status_clean
from tests.util import TOL, assert_close, bits_equal, to_np

pytestmark = pytest.mark.gpu


def _sub_pool(pool_dev, idx):
    """CPU copy of the slots idx refers to, and idx remapped onto it."""
    idx = idx.to(torch.int64)
    live = idx >= 0
    sub = pool_dev[idx.clamp(min=0).to(DEV)].cpu()
    local = torch.where(live, torch.arange(len(idx)), torch.full_like(idx, -1))
    return sub, local.numpy()


def _state_err(pool_dev, upd, where):
    """max |gpu - oracle| / max |oracle| over the states in upd; where(key)
    gives the (slot, head) of the GPU pool that holds key's state."""
    num = den = 0.0
    for key, S in upd.items():
        slot, h = where(key)
        got = pool_dev[slot, h].cpu().double().numpy()
        num = max(num, float(np.abs(got - S).max()))
        den = max(den, float(np.abs(S).max()))
    return num / den


def _untouched(pool_dev, before_dev, touched):
    mask = torch.ones(pool_dev.shape[0], dtype=torch.bool, device=DEV)
    if touched:
        mask[torch.tensor(sorted(touched), device=DEV)] = False
    a = pool_dev[mask].view(torch.int32)
    b = before_dev[mask].view(torch.int32)
    return bool(torch.equal(a, b))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_decode_full_size(dtype):
    """256 sequences x 1 token, 16 QK / 32 V heads, dk = dv = 128, pool of
    1024 slots ~ N(0, 0.02), slots a seeded permutation subset; one padding row."""
    w = workloads.decode(dtype=dtype, pool_device=DEV)
    pool = w.state_pool
    before = pool.clone()
    idx = w.slots.clone()
    pad_slot = int(idx[3])
    idx[3] = -1
    q, k, v, a, b = (cuda(t) for t in (w.q, w.k, w.v, w.a, w.b))
    g, beta = gdn().gdn_gating(a, b, cuda(w.A_log), cuda(w.dt_bias))
    o = gdn().gdn_decode_recurrent(q, k, v, g, beta, 1, pool, cuda(idx), scale=w.scale)
    torch.cuda.synchronize()
    status_clean()

    g_ref, b_ref = oracle_gating(w.a, w.b, w.A_log, w.dt_bias)
    sub, local = _sub_pool(before, idx)
    o_ref, upd = oracle.gdn_decode(to_np(w.q), to_np(w.k), to_np(w.v), g_ref, b_ref, 1, sub, local,
                                   scale=w.scale)
    assert_close(o, o_ref, TOL[dtype], "decode o")
    assert torch.all(o[3] == 0)
    err = _state_err(pool, upd, lambda key: (int(idx[key[0]]), key[1]))
    assert err <= TOL[dtype], f"decode state rel err {err:.3e}"
    assert _untouched(pool, before, {int(s) for s in idx if s >= 0})
    assert bits_equal(pool[pad_slot], before[pad_slot])


def test_decode_layer_chain_full_size():
    """conv update -> q/k/v views of its output (row stride 8192) -> gating ->
    decode, against the same chain in the oracle."""
    w = workloads.decode(pool_device=DEV)
    d = w.dims
    pool, before = w.state_pool, w.state_pool.clone()
    cpool = cuda(w.conv_pool)
    idx = cuda(w.slots)
    y = gdn().causal_conv1d_update(cuda(w.x), 1, cuda(w.conv_w), cpool, idx)
    qv, kv, vv = qkv_views(y, d)
    g, beta = gdn().gdn_gating(cuda(w.a), cuda(w.b), cuda(w.A_log), cuda(w.dt_bias))
    o = gdn().gdn_decode_recurrent(qv, kv, vv, g, beta, 1, pool, idx, scale=w.scale)
    torch.cuda.synchronize()
    status_clean()

    y_ref, _ = oracle.conv1d_update(to_np(w.x), 1, to_np(w.conv_w), None, to_np(w.conv_pool),
                                    to_np(w.slots).astype(np.int64))
    q_r, k_r, v_r = oracle.split_qkv(y_ref, d.hqk, d.hv, d.dk, d.dv)
    g_ref, b_ref = oracle_gating(w.a, w.b, w.A_log, w.dt_bias)
    sub, local = _sub_pool(before, w.slots)
    o_ref, upd = oracle.gdn_decode(q_r, k_r, v_r, g_ref, b_ref, 1, sub, local, scale=w.scale)
    assert_close(o, o_ref, TOL[torch.bfloat16], "chained decode o")
    err = _state_err(pool, upd, lambda key: (int(w.slots[key[0]]), key[1]))
    assert err <= TOL[torch.bfloat16], f"chained decode state rel err {err:.3e}"


def test_mtp_full_size_snapshots_and_accept():
    """128 sequences x 4 tokens; after token t the state goes to snap[i][t];
    the source slot and every other slot stay bit-identical; accepting draft
    token a[i] copies snap[i][a[i]] into the source slot bit for bit."""
    w = workloads.mtp(pool_device=DEV)
    pool, before = w.state_pool, w.state_pool.clone()
    q, k, v, a, b = (cuda(t) for t in (w.q, w.k, w.v, w.a, w.b))
    snap = cuda(w.snap)
    g, beta = gdn().gdn_gating(a, b, cuda(w.A_log), cuda(w.dt_bias))
    o = gdn().gdn_decode_recurrent(q, k, v, g, beta, 4, pool, cuda(w.slots), snap, scale=w.scale)
    torch.cuda.synchronize()
    status_clean()

    g_ref, b_ref = oracle_gating(w.a, w.b, w.A_log, w.dt_bias)
    sub, local = _sub_pool(before, w.slots)
    snap_local = np.arange(w.n_seqs * 4).reshape(w.n_seqs, 4) + 10_000     # tags, remapped below
    o_ref, upd = oracle.gdn_decode(to_np(w.q), to_np(w.k), to_np(w.v), g_ref, b_ref, 4, sub, local,
                                   snap_local, scale=w.scale)
    assert_close(o, o_ref, TOL[torch.bfloat16], "mtp o")
    snap_np = w.snap.numpy()

    def where(key):
        i, t = divmod(key[0] - 10_000, 4)
        return int(snap_np[i, t]), key[1]
    err = _state_err(pool, upd, where)
    assert err <= TOL[torch.bfloat16], f"mtp snapshot rel err {err:.3e}"
    assert _untouched(pool, before, set(snap_np.reshape(-1).tolist()))

    # accept: slot[i] <- snap[i][accept[i]]
    acc = w.extra["accept"].long()
    src = w.snap[torch.arange(w.n_seqs), acc].to(torch.int32)
    gdn().gdn_state_snapshot(pool, cuda(src), cuda(w.slots))
    torch.cuda.synchronize()
    status_clean()
    assert bits_equal(pool[w.slots.long().to(DEV)], pool[src.long().to(DEV)])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,dv,tps", [(16, 16, 1), (16, 24, 3), (32, 32, 2), (64, 128, 16),
                                       (128, 64, 5), (128, 128, 1), (128, 128, 4), (128, 128, 16)])
def test_decode_small_shapes(dtype, dk, dv, tps):
    gen = torch.Generator().manual_seed(dk * 1000 + dv * 10 + tps)
    hqk, hv, N, slots = 2, 4, 5, 12
    T = N * tps
    q = torch.randn(T, hqk, dk, generator=gen).to(dtype)
    k = torch.randn(T, hqk, dk, generator=gen).to(dtype)
    v = torch.randn(T, hv, dv, generator=gen).to(dtype)
    a = torch.randn(T, hv, generator=gen).to(dtype)
    b = torch.randn(T, hv, generator=gen).to(dtype)
    A_log, dt_bias = workloads.gating_params(gen, hv, low_decay=True)
    pool = torch.randn(slots, hv, dv, dk, generator=gen) * 0.1
    idx = torch.tensor([4, 0, -1, 11, 7], dtype=torch.int32)
    snap = None
    if tps > 1:                       # destinations 1, 2, 3, 5 are never sources
        snap = torch.full((N, tps), -1, dtype=torch.int32)
        snap[1, 0], snap[1, tps - 1], snap[4, 0], snap[0, tps - 1] = 1, 2, 3, 5
    pd = cuda(pool)
    g, beta = gdn().gdn_gating(cuda(a), cuda(b), cuda(A_log), cuda(dt_bias))
    o = gdn().gdn_decode_recurrent(cuda(q), cuda(k), cuda(v), g, beta, tps, pd, cuda(idx),
                                   cuda(snap), scale=0.3)
    torch.cuda.synchronize()
    status_clean()
    g_ref, b_ref = oracle_gating(a, b, A_log, dt_bias)
    o_ref, upd = oracle.gdn_decode(to_np(q), to_np(k), to_np(v), g_ref, b_ref, tps, to_np(pool),
                                   to_np(idx).astype(np.int64),
                                   None if snap is None else to_np(snap).astype(np.int64), scale=0.3)
    assert_close(o, o_ref, TOL[dtype], "o")
    got = pd.cpu()
    for s in range(slots):
        for h in range(hv):
            if (s, h) in upd:
                assert_close(got[s, h], upd[(s, h)], TOL[dtype], f"state {s},{h}")
            else:
                assert bits_equal(got[s, h], pool[s, h]), f"untouched {s},{h}"


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_decode_multitoken_in_place(dtype):
    """dk = dv = 128, 3 tokens per sequence and no snapshots: the state is
    updated in its own slot after the last token; a padding row is skipped."""
    gen = torch.Generator().manual_seed(77)
    hqk, hv, N, tps, slots = 2, 4, 6, 3, 9
    T = N * tps
    q = torch.randn(T, hqk, 128, generator=gen).to(dtype)
    k = torch.randn(T, hqk, 128, generator=gen).to(dtype)
    v = torch.randn(T, hv, 128, generator=gen).to(dtype)
    a = torch.randn(T, hv, generator=gen).to(dtype)
    b = torch.randn(T, hv, generator=gen).to(dtype)
    A_log, dt_bias = workloads.gating_params(gen, hv, low_decay=True)
    pool = torch.randn(slots, hv, 128, 128, generator=gen) * 0.05
    idx = torch.tensor([8, 2, -1, 0, 5, 3], dtype=torch.int32)
    pd = cuda(pool)
    g, beta = gdn().gdn_gating(cuda(a), cuda(b), cuda(A_log), cuda(dt_bias))
    o = gdn().gdn_decode_recurrent(cuda(q), cuda(k), cuda(v), g, beta, tps, pd, cuda(idx), scale=0.2)
    torch.cuda.synchronize()
    status_clean()
    g_ref, b_ref = oracle_gating(a, b, A_log, dt_bias)
    o_ref, upd = oracle.gdn_decode(to_np(q), to_np(k), to_np(v), g_ref, b_ref, tps, to_np(pool),
                                   to_np(idx).astype(np.int64), None, scale=0.2)
    assert_close(o, o_ref, TOL[dtype], "o")
    assert torch.all(o[2 * tps:3 * tps] == 0)
    got = pd.cpu()
    for s in range(slots):
        for h in range(hv):
            if (s, h) in upd:
                assert_close(got[s, h], upd[(s, h)], TOL[dtype], f"state {s},{h}")
            else:
                assert bits_equal(got[s, h], pool[s, h]), f"untouched {s},{h}"


def test_decode_bad_slot_flags_status():
    """A slot index >= n_slots is skipped (zero output, nothing written) and
    reported in the device status word."""
    gen = torch.Generator().manual_seed(5)
    q = torch.randn(2, 1, 16, generator=gen)
    k = torch.randn(2, 1, 16, generator=gen)
    v = torch.randn(2, 2, 16, generator=gen)
    g = -torch.rand(2, 2, generator=gen)
    beta = torch.rand(2, 2, generator=gen)
    pool = torch.randn(3, 2, 16, 16, generator=gen)
    pd = cuda(pool)
    idx = torch.tensor([1, 3], dtype=torch.int32)           # 3 is out of range
    gdn().gdn_get_device_status(clear=True)
    o = gdn().gdn_decode_recurrent(cuda(q), cuda(k), cuda(v), cuda(g), cuda(beta), 1, pd,
                                   cuda(idx), scale=1.0)
    st = gdn().gdn_get_device_status(clear=True)
    assert st & gdn().DEVSTAT_BAD_INDEX
    assert torch.all(o[1] == 0)
    assert bits_equal(pd.cpu()[0], pool[0]) and bits_equal(pd.cpu()[2], pool[2])
    assert gdn().gdn_get_device_status(clear=True) == 0
