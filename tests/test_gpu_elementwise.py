"""GPU parity of the elementwise passes (gating, conv1d fwd / update) and of
the whole-slot snapshot copy, through the C ABI, against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_common import DEV, cuda, gdn, oracle_gating, status_clean
from tests.util import TOL, assert_close, bits_equal, to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,hv", [(256, 32), (1, 4), (37, 32), (0, 32)])
def test_gating(dtype, T, hv):
    gen = torch.Generator().manual_seed(T * 7 + hv)
    a = (torch.randn(T, hv, generator=gen) * 3).to(dtype)
    b = (torch.randn(T, hv, generator=gen) * 3).to(dtype)
    if T:
        a[0, :4] = torch.tensor([80.0, -80.0, 19.9, 20.1]).to(dtype)
        b[0, :4] = torch.tensor([80.0, -80.0, 0.0, 1.0]).to(dtype)
    A_log, dt_bias = workloads.gating_params(gen, hv)
    g, beta = gdn().gdn_gating(cuda(a), cuda(b), cuda(A_log), cuda(dt_bias))
    torch.cuda.synchronize()
    status_clean()
    if T == 0:
        assert g.numel() == 0
        return
    g_ref, b_ref = oracle_gating(a, b, A_log, dt_bias)
    np.testing.assert_allclose(to_np(g), g_ref, rtol=2e-6, atol=1e-30)
    np.testing.assert_allclose(to_np(beta), b_ref, rtol=2e-6, atol=1e-30)


def _conv_oracle(x, cu, w, pool, idx, has, bias=None):
    y, upd = oracle.conv1d_fwd(to_np(x), to_np(cu).astype(np.int64), to_np(w),
                               None if bias is None else to_np(bias),
                               pool, to_np(idx).astype(np.int64),
                               None if has is None else to_np(has).astype(np.int64))
    return y, upd


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_conv_fwd_varlen_ragged(dtype):
    """Sequences of 0, 1, 2, 3, 17, 40 tokens spanning several token runs;
    slots with / without history, padding slot -1; a strided x view."""
    gen = torch.Generator().manual_seed(11)
    C, W = 256, 4
    lens = [17, 0, 1, 2, 40, 3]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    T = int(cu[-1])
    xbig = torch.randn(T, C + 64, generator=gen).to(dtype)
    x = xbig[:, 32:32 + C]                            # row stride C + 64
    w = workloads.conv_weight(gen, C, W, dtype)
    pool = torch.randn(8, W - 1, C, generator=gen).to(dtype)
    idx = torch.tensor([3, 1, -1, 5, 0, 6], dtype=torch.int32)
    has = torch.tensor([1, 1, 1, 0, 1, 1], dtype=torch.uint8)
    xd, pd = cuda(xbig)[:, 32:32 + C], cuda(pool)
    y = gdn().causal_conv1d_fwd(xd, cuda(w), cuda(cu), pd, cuda(idx), cuda(has))
    torch.cuda.synchronize()
    status_clean()
    y_ref, upd = _conv_oracle(x, cu, w, to_np(pool), idx, has)
    assert_close(y, y_ref, TOL[dtype], "conv y")
    got = pd.cpu()
    for s in range(8):
        if s in upd:
            ref = torch.from_numpy(upd[s]).to(dtype)
            assert bits_equal(got[s], ref), f"conv state slot {s}"    # states are copies of inputs
        else:
            assert bits_equal(got[s], pool[s]), f"untouched slot {s}"


@pytest.mark.parametrize("W", [2, 3, 4])
def test_conv_fwd_tma_ragged(W):
    """The TMA-staged path (bf16, channels a multiple of 512): 1024 channels,
    138 tokens in tiles of 32 with sequence starts inside tiles, empty
    sequences at the start, inside a tile and at a tile edge, sequences of
    1..3 tokens, slots with / without history, a padding slot, a strided x
    view, a conv bias and a ragged last tile."""
    gen = torch.Generator().manual_seed(12 + W)
    C = 1024
    lens = [0, 17, 0, 1, 2, 12, 0, 40, 3, 0, 58, 5]
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    T = int(cu[-1])
    xbig = torch.randn(T, C + 64, generator=gen).to(torch.bfloat16)
    x = xbig[:, 32:32 + C]                            # row stride C + 64
    w = workloads.conv_weight(gen, C, W, torch.bfloat16)
    bias = (torch.randn(C, generator=gen) * 0.1).to(torch.bfloat16)
    pool = torch.randn(14, W - 1, C, generator=gen).to(torch.bfloat16)
    idx = torch.tensor([9, 3, 1, -1, 5, 11, 12, 0, 6, 8, 2, 13], dtype=torch.int32)
    has = torch.tensor([1, 1, 1, 1, 0, 1, 1, 1, 1, 1, 0, 1], dtype=torch.uint8)
    xd, pd = cuda(xbig)[:, 32:32 + C], cuda(pool)
    y = gdn().causal_conv1d_fwd(xd, cuda(w), cuda(cu), pd, cuda(idx), cuda(has), bias=cuda(bias))
    torch.cuda.synchronize()
    status_clean()
    y_ref, upd = _conv_oracle(x, cu, w, to_np(pool), idx, has, bias)
    assert_close(y, y_ref, TOL[torch.bfloat16], "conv y (TMA path)")
    got = pd.cpu()
    for s in range(pool.shape[0]):
        if s in upd:
            assert bits_equal(got[s], torch.from_numpy(upd[s]).to(torch.bfloat16)), f"slot {s}"
        else:
            assert bits_equal(got[s], pool[s]), f"untouched slot {s}"


def test_conv_fwd_full_prefill_sampled_channels():
    """Full prefill batch (8 sequences, 512..8192 tokens, 8192 channels); the
    oracle recomputes 384 sampled channels (each channel is independent)."""
    w = workloads.prefill()
    xd = cuda(w.x)
    pool = cuda(w.conv_pool)
    y = gdn().causal_conv1d_fwd(xd, cuda(w.conv_w), cuda(w.cu_seqlens), pool, cuda(w.slots),
                                cuda(w.has_initial_state))
    torch.cuda.synchronize()
    status_clean()
    rng = np.random.default_rng(0)
    ch = np.sort(np.concatenate([[0, 7, 2047, 2048, 4095, 4096, 8191],
                                 rng.choice(8192, 377, replace=False)]))
    ch = np.unique(ch)
    xs = to_np(w.x[:, ch])
    y_ref, upd = oracle.conv1d_fwd(xs, to_np(w.cu_seqlens).astype(np.int64), to_np(w.conv_w)[ch],
                                   None, to_np(w.conv_pool)[:, :, ch],
                                   to_np(w.slots).astype(np.int64),
                                   to_np(w.has_initial_state).astype(np.int64))
    assert_close(y[:, ch], y_ref, TOL[torch.bfloat16], "conv y (sampled)")
    got = pool.cpu()
    for s, st in upd.items():
        assert bits_equal(got[s][:, ch], torch.from_numpy(st).to(torch.bfloat16))


@pytest.mark.parametrize("tps,use_snap", [(1, False), (4, True), (4, False)])
def test_conv_update(tps, use_snap):
    """Decode (256 x 1) and MTP (128 x 4, with per-token conv snapshots)."""
    w = workloads.decode() if tps == 1 else workloads.mtp()
    x = w.x[: w.n_seqs * tps]
    idx = w.slots.clone()
    idx[5] = -1                                          # one padding row
    snap = w.snap if use_snap else None
    pool = cuda(w.conv_pool)
    y = gdn().causal_conv1d_update(cuda(x), tps, cuda(w.conv_w), pool, cuda(idx), cuda(snap))
    torch.cuda.synchronize()
    status_clean()
    y_ref, upd = oracle.conv1d_update(to_np(x), tps, to_np(w.conv_w), None, to_np(w.conv_pool),
                                      to_np(idx).astype(np.int64),
                                      None if snap is None else to_np(snap).astype(np.int64))
    assert_close(y, y_ref, TOL[torch.bfloat16], "conv update y")
    assert torch.all(y[5 * tps:6 * tps] == 0)
    got = pool.cpu()
    touched = set(upd)
    for s, st in upd.items():
        assert bits_equal(got[s], torch.from_numpy(st).to(torch.bfloat16)), f"slot {s}"
    for s in range(got.shape[0]):
        if s not in touched:
            assert bits_equal(got[s], w.conv_pool[s]), f"untouched slot {s}"


def test_state_snapshot_bit_exact():
    gen = torch.Generator().manual_seed(3)
    pool = torch.randn(16, 4, 8, 8, generator=gen)
    pool[2, 0, 0, 0] = float("nan")
    src = torch.tensor([2, 5, -1, 9], dtype=torch.int32)
    dst = torch.tensor([7, 1, 3, -1], dtype=torch.int32)
    pd = cuda(pool)
    gdn().gdn_state_snapshot(pd, cuda(src), cuda(dst))
    torch.cuda.synchronize()
    status_clean()
    got = pd.cpu()
    upd = oracle.state_snapshot(to_np(pool), to_np(src).astype(np.int64), to_np(dst).astype(np.int64))
    for s in range(16):
        want = pool[2] if s == 7 else pool[5] if s == 1 else pool[s]
        assert bits_equal(got[s], want), s
    assert set(upd) == {7, 1}
    # bf16 conv-state pool (slot of 3 x 8192 x 2 bytes)
    cp = torch.randn(6, 3, 8192, generator=gen).to(torch.bfloat16)
    cpd = cuda(cp)
    gdn().gdn_state_snapshot(cpd, cuda(torch.tensor([0], dtype=torch.int32)),
                             cuda(torch.tensor([4], dtype=torch.int32)))
    torch.cuda.synchronize()
    assert bits_equal(cpd.cpu()[4], cp[0]) and bits_equal(cpd.cpu()[0], cp[0])
