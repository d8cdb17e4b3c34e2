"""GPU parity of the fused MTP step (conv update with per-token conv
snapshots, gating, L2 norms and the multi-token recurrent update with
per-token state snapshots, in one kernel) through the C ABI, against the
oracle's conv update -> gating -> decode chain with the same snapshots: o
and the snapshot states within the bf16 tolerance, the conv snapshots bit for
bit, the source slots and every other slot unchanged; at the full MTP size
(128 sequences x 4 tokens, with a padding row and a skipped snapshot) and at
small shapes with a conv bias (GQA 1, 2 and 3, 1 to 16 tokens, an unaligned x
row stride); and against the three-call path."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_common import DEV, cuda, gdn, oracle_gating, status_clean
from tests.util import TOL, assert_close, bits_equal, to_np
from tests.test_gpu_decode import _state_err, _sub_pool, _untouched

pytestmark = pytest.mark.gpu


def _check_mtp(x, tps, conv_w, conv_b, cpool0, a, b, A_log, dt_bias, pool0, idx, snap, hqk, hv,
               scale, x_pad=0):
    cpool = cuda(cpool0)
    pool = cuda(pool0)
    # x_pad > 0: x as the first C columns of wider rows (a row stride that is
    # not a multiple of 16 bytes takes the element-by-element staging)
    xd = cuda(torch.nn.functional.pad(x, (0, x_pad)))[:, :x.shape[1]] if x_pad else cuda(x)
    o = gdn().gdn_mtp_step_fused(xd, tps, cuda(conv_w), cpool, cuda(a), cuda(b),
                                 cuda(A_log), cuda(dt_bias), hqk, pool, cuda(idx), cuda(snap),
                                 scale=scale, conv_bias=None if conv_b is None else cuda(conv_b))
    torch.cuda.synchronize()
    status_clean()
    idx64 = to_np(idx).astype(np.int64)
    y_ref, conv_upd = oracle.conv1d_update(to_np(x), tps, to_np(conv_w),
                                           None if conv_b is None else to_np(conv_b),
                                           to_np(cpool0), idx64, snap_indices=to_np(snap))
    q_r, k_r, v_r = oracle.split_qkv(y_ref, hqk, hv, 128, 128)
    g_ref, b_ref = oracle_gating(a, b, A_log, dt_bias)
    live = idx >= 0
    snap_local = torch.where(live[:, None], snap, torch.full_like(snap, -1))
    sub, local = _sub_pool(cuda(pool0), idx)
    o_ref, upd = oracle.gdn_decode(q_r, k_r, v_r, g_ref, b_ref, tps, sub, local,
                                   snap_indices=to_np(snap_local).astype(np.int64), scale=scale)
    assert_close(o, o_ref, TOL[torch.bfloat16], "fused MTP o")
    dead_rows = (~live).repeat_interleave(tps)
    assert torch.all(o[dead_rows.to(DEV)] == 0)
    err = _state_err(pool, upd, lambda key: key)
    assert err <= TOL[torch.bfloat16], f"fused MTP snapshot state rel err {err:.3e}"
    assert _untouched(pool, cuda(pool0), {s for (s, _h) in upd})
    got = cpool.cpu()
    for s, st in conv_upd.items():
        assert bits_equal(got[s], torch.from_numpy(st).to(torch.bfloat16)), f"conv slot {s}"
    others = torch.ones(cpool0.shape[0], dtype=torch.bool)
    if conv_upd:
        others[torch.tensor(sorted(conv_upd), dtype=torch.long)] = False
    assert bits_equal(got[others], cpool0[others])
    return o, pool, cpool


def test_fused_mtp_full_size():
    """128 sequences x 4 tokens, 16 QK / 32 V heads, pools of 1024 slots;
    sequence 9 has no slot, one snapshot entry is skipped."""
    w = workloads.mtp()
    d = w.dims
    idx = w.slots.clone()
    idx[9] = -1
    snap = w.snap.clone()
    snap[3, 2] = -1
    _check_mtp(w.x, 4, w.conv_w, None, w.conv_pool, w.a, w.b, w.A_log, w.dt_bias,
               w.state_pool, idx, snap, d.hqk, d.hv, w.scale)


@pytest.mark.parametrize("hqk,hv,tps,x_pad", [(2, 4, 4, 0), (4, 4, 3, 0), (1, 2, 1, 0),
                                              (2, 4, 5, 3), (1, 3, 16, 0)])
def test_fused_mtp_small_with_bias(hqk, hv, tps, x_pad):
    g = torch.Generator().manual_seed(71 + 10 * hv + tps)
    n = 6
    n_slots = n * (tps + 1) + 3
    C = 2 * hqk * 128 + hv * 128
    x = torch.randn(n * tps, C, generator=g).bfloat16()
    conv_w = (torch.rand(C, 4, generator=g) - 0.5).bfloat16()
    conv_b = (torch.randn(C, generator=g) * 0.1).bfloat16()
    cpool0 = torch.randn(n_slots, 3, C, generator=g).bfloat16()
    a = torch.randn(n * tps, hv, generator=g).bfloat16()
    b = torch.randn(n * tps, hv, generator=g).bfloat16()
    A_log, dt_bias = workloads.gating_params(g, hv, False)
    pool0 = torch.randn(n_slots, hv, 128, 128, generator=g) * 0.02
    perm = torch.randperm(n_slots, generator=g).to(torch.int32)
    idx = perm[:n].clone()
    idx[2] = -1
    snap = perm[n:n + n * tps].view(n, tps).clone()
    _check_mtp(x, tps, conv_w, conv_b, cpool0, a, b, A_log, dt_bias, pool0, idx, snap, hqk, hv,
               128 ** -0.5, x_pad)


def test_fused_mtp_matches_three_calls():
    """The fused step against causal_conv1d_update + gdn_gating +
    gdn_decode_recurrent with the same snapshots on the MTP workload: o
    within 1e-2 of max|o| (the fused kernel keeps q, k, v in fp32 where the
    three calls round them to bf16), conv snapshots bit for bit."""
    w = workloads.mtp(pool_device=DEV)
    d = w.dims
    x, a, b = cuda(w.x), cuda(w.a), cuda(w.b)
    conv_w, A_log, dt_bias = cuda(w.conv_w), cuda(w.A_log), cuda(w.dt_bias)
    slots, snap = cuda(w.slots), cuda(w.snap)
    c1, c2 = cuda(w.conv_pool), cuda(w.conv_pool)
    p1, p2 = w.state_pool.clone(), w.state_pool.clone()
    o1 = gdn().gdn_mtp_step_fused(x, 4, conv_w, c1, a, b, A_log, dt_bias, d.hqk, p1, slots, snap,
                                  scale=w.scale)
    y = gdn().causal_conv1d_update(x, 4, conv_w, c2, slots, snap_indices=snap)
    nq = d.hqk * d.dk
    q = y.narrow(1, 0, nq).unflatten(1, (d.hqk, d.dk))
    k = y.narrow(1, nq, nq).unflatten(1, (d.hqk, d.dk))
    v = y.narrow(1, 2 * nq, d.hv * d.dv).unflatten(1, (d.hv, d.dv))
    g, beta = gdn().gdn_gating(a, b, A_log, dt_bias)
    o2 = gdn().gdn_decode_recurrent(q, k, v, g, beta, 4, p2, slots, snap_indices=snap,
                                    scale=w.scale)
    torch.cuda.synchronize()
    status_clean()
    assert_close(o1, o2, 1e-2, "fused vs three calls: o")
    sn = w.snap.view(-1).long()
    assert_close(p1[sn.to(DEV)], p2[sn.to(DEV)], 1e-2, "fused vs three calls: snapshots")
    assert bits_equal(c1, c2), "conv pools differ"
    assert bits_equal(p1[w.slots.long().to(DEV)], w.state_pool[w.slots.long().to(DEV)])
