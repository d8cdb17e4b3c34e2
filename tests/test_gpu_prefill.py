"""GPU parity of the chunked varlen prefill through the C ABI against the CPU
oracle: the tiny fp32 layer (conv -> gating -> prefill), a sweep of head
sizes / chunks / ragged lengths with initial states, the full 8-sequence
prefill layer on sampled (sequence, head) chains, and the 65536-token
sequence with split-and-carry."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_common import DEV, cuda, gdn, oracle_gating, qkv_views, status_clean
from tests.util import TOL, assert_close, bits_equal, to_np

pytestmark = pytest.mark.gpu


def test_tiny_fp32_layer():
    """1 sequence, T = 64, 2 QK / 4 V heads, head_dim 16, conv width 4 over 128
    channels, chunk 16, zero initial state, fp32: o, final state, conv state."""
    w = workloads.tiny()
    d = w.dims
    cpool = cuda(w.conv_pool)
    spool = cuda(w.state_pool)
    slots = cuda(w.slots)
    y = gdn().causal_conv1d_fwd(cuda(w.x), cuda(w.conv_w), cuda(w.cu_seqlens), cpool, slots,
                                cuda(w.has_initial_state))
    q, k, v = qkv_views(y, d)
    g, beta = gdn().gdn_gating(cuda(w.a), cuda(w.b), cuda(w.A_log), cuda(w.dt_bias))
    init = torch.where(w.has_initial_state.bool(), w.slots, torch.full_like(w.slots, -1))
    o = gdn().gdn_prefill_chunked(q, k, v, g, beta, cuda(w.cu_seqlens), spool, cuda(init), slots,
                                  w.scale, chunk=w.chunk)
    torch.cuda.synchronize()
    status_clean()
    o_ref, conv_upd, upd, g_ref, b_ref, y_ref = oracle.layer_prefill(
        w.x, w.cu_seqlens, w.conv_w, None, w.conv_pool, w.A_log, w.dt_bias, w.a, w.b,
        w.state_pool, w.slots, w.has_initial_state, d.hqk, d.hv, d.dk, d.dv, w.scale)
    assert_close(y, y_ref, 1e-5, "conv y")
    assert_close(g, g_ref, 1e-5, "g")
    assert_close(o, o_ref, TOL[torch.float32], "o")
    got = spool.cpu()
    for (s, h), S in upd.items():
        assert_close(got[s, h], S, TOL[torch.float32], f"final state {s},{h}")
    for s, st in conv_upd.items():
        assert bits_equal(cpool.cpu()[s], torch.from_numpy(st).float())


def _direct_batch(seed, lens, hqk, hv, dk, dtype, low_decay, n_slots=8):
    gen = torch.Generator().manual_seed(seed)
    T = sum(lens)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    q = torch.randn(T, hqk, dk, generator=gen).to(dtype)
    k = torch.randn(T, hqk, dk, generator=gen).to(dtype)
    v = torch.randn(T, hv, dk, generator=gen).to(dtype)
    a = torch.randn(T, hv, generator=gen).to(dtype)
    b = torch.randn(T, hv, generator=gen).to(dtype)
    A_log, dt_bias = workloads.gating_params(gen, hv, low_decay)
    pool = torch.randn(n_slots, hv, dk, dk, generator=gen) * 0.05
    return cu, q, k, v, a, b, A_log, dt_bias, pool


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dk,chunk", [(16, 16), (32, 32), (64, 64), (128, 64), (128, 16),
                                      (64, 16), (128, 32)])
@pytest.mark.parametrize("low_decay", [False, True])
def test_prefill_sweep(dtype, dk, chunk, low_decay):
    """Ragged lengths (0, 1, chunk-1, chunk, chunk+1, 3 chunks + 7), nonzero
    initial states (one zero-init, one in-place carry), GQA 2 -> 4 heads."""
    lens = [chunk + 1, 0, 1, chunk - 1, chunk, 3 * chunk + 7]
    hqk, hv = 2, 4
    cu, q, k, v, a, b, A_log, dt_bias, pool = _direct_batch(dk * 7 + chunk + low_decay, lens, hqk,
                                                            hv, dk, dtype, low_decay)
    init = torch.tensor([0, 1, -1, 3, 4, 5], dtype=torch.int32)
    final = torch.tensor([6, 7, 2, 3, -1, 5], dtype=torch.int32)
    pd = cuda(pool)
    g, beta = gdn().gdn_gating(cuda(a), cuda(b), cuda(A_log), cuda(dt_bias))
    o = gdn().gdn_prefill_chunked(cuda(q), cuda(k), cuda(v), g, beta, cuda(cu), pd, cuda(init),
                                  cuda(final), 0.25, chunk=chunk)
    torch.cuda.synchronize()
    status_clean()
    g_ref, b_ref = oracle_gating(a, b, A_log, dt_bias)
    o_ref, upd, _ = oracle.gdn_prefill(to_np(q), to_np(k), to_np(v), g_ref, b_ref, to_np(cu),
                                       to_np(pool), to_np(init), to_np(final), 0.25)
    assert_close(o, o_ref, TOL[dtype], "o")
    got = pd.cpu()
    for s in range(pool.shape[0]):
        for h in range(hv):
            if (s, h) in upd:
                assert_close(got[s, h], upd[(s, h)], TOL[dtype], f"state {s},{h}")
            else:
                assert bits_equal(got[s, h], pool[s, h]), f"untouched {s},{h}"


@pytest.mark.parametrize("workspace", [None, False], ids=["split", "fused"])
@pytest.mark.parametrize("low_decay", [False, True])
def test_prefill_tc_paths(workspace, low_decay):
    """bf16, dk = dv = 128, chunk 64: the two-kernel path (prep kernel +
    chain kernel, workspace given) and the single fused kernel (no
    workspace).  Ragged lengths up to 10 chunks so that every stage ring
    wraps, nonzero initial states, GQA 2 -> 4 heads."""
    lens = [65, 0, 1, 63, 64, 199, 9 * 64 + 13, 2]
    hqk, hv, dk = 2, 4, 128
    cu, q, k, v, a, b, A_log, dt_bias, pool = _direct_batch(4242 + low_decay, lens, hqk, hv, dk,
                                                            torch.bfloat16, low_decay, n_slots=10)
    init = torch.tensor([0, 1, -1, 3, 4, 5, 8, 9], dtype=torch.int32)
    final = torch.tensor([6, 7, 2, 3, -1, 5, 8, -1], dtype=torch.int32)
    pd = cuda(pool)
    g, beta = gdn().gdn_gating(cuda(a), cuda(b), cuda(A_log), cuda(dt_bias))
    o = gdn().gdn_prefill_chunked(cuda(q), cuda(k), cuda(v), g, beta, cuda(cu), pd, cuda(init),
                                  cuda(final), 0.125, chunk=64, workspace=workspace)
    torch.cuda.synchronize()
    status_clean()
    g_ref, b_ref = oracle_gating(a, b, A_log, dt_bias)
    o_ref, upd, _ = oracle.gdn_prefill(to_np(q), to_np(k), to_np(v), g_ref, b_ref, to_np(cu),
                                       to_np(pool), to_np(init), to_np(final), 0.125)
    assert_close(o, o_ref, TOL[torch.bfloat16], "o")
    got = pd.cpu()
    for s in range(pool.shape[0]):
        for h in range(hv):
            if (s, h) in upd:
                assert_close(got[s, h], upd[(s, h)], TOL[torch.bfloat16], f"state {s},{h}")
            else:
                assert bits_equal(got[s, h], pool[s, h]), f"untouched {s},{h}"


def test_prefill_empty_batch_and_all_empty_sequences():
    hv, dk = 4, 16
    pool = torch.randn(3, hv, dk, dk)
    pd = cuda(pool)
    cu = cuda(torch.zeros(3, dtype=torch.int32))
    z = torch.zeros(0, 2, dk, device=DEV)
    zv = torch.zeros(0, hv, dk, device=DEV)
    g = torch.zeros(0, hv, device=DEV)
    o = gdn().gdn_prefill_chunked(z, z, zv, g, g, cu, pd, cuda(torch.tensor([0, -1], dtype=torch.int32)),
                                  cuda(torch.tensor([1, 2], dtype=torch.int32)), 1.0, chunk=16)
    torch.cuda.synchronize()
    status_clean()
    got = pd.cpu()
    assert o.numel() == 0
    assert bits_equal(got[1], pool[0])            # empty sequence carries its state
    assert torch.all(got[2] == 0)                 # zero init, nothing seen: zero state


def _oracle_chain_from_x(w, seq, h):
    """Oracle: conv over the 3 x 128 channels one (sequence, V head) chain
    reads, SiLU, gating of head h, token recurrence."""
    d = w.dims
    hq = h // (d.hv // d.hqk)
    nq = d.hqk * d.dk
    ch = np.concatenate([np.arange(hq * d.dk, (hq + 1) * d.dk),
                         nq + np.arange(hq * d.dk, (hq + 1) * d.dk),
                         2 * nq + np.arange(h * d.dv, (h + 1) * d.dv)])
    s, e = int(w.cu_seqlens[seq]), int(w.cu_seqlens[seq + 1])
    y, _ = oracle.conv1d_seq(to_np(w.x[s:e][:, ch]), to_np(w.conv_w)[ch])
    g, beta = oracle.gating(to_np(w.a[s:e, h:h + 1]), to_np(w.b[s:e, h:h + 1]),
                            to_np(w.A_log[h:h + 1]), to_np(w.dt_bias[h:h + 1]))
    return oracle.recurrent_chain(y[:, :d.dk], y[:, d.dk:2 * d.dk], y[:, 2 * d.dk:], g[:, 0],
                                  beta[:, 0], scale=w.scale)


@pytest.mark.parametrize("workspace", [None, False], ids=["split", "fused"])
def test_prefill_full_layer_sampled_chains(workspace):
    """8 sequences, lengths U{512..8192}: conv -> gating -> prefill on the GPU
    (two-kernel and fused paths); the oracle recomputes 24 (sequence, head)
    chains end to end from x, three per sequence."""
    w = workloads.prefill()
    d = w.dims
    cpool = cuda(w.conv_pool)
    spool = torch.zeros((64, d.hv, d.dv, d.dk), device=DEV)
    slots = (w.slots % 64).to(torch.int32)
    none = torch.full_like(slots, -1)
    y = gdn().causal_conv1d_fwd(cuda(w.x), cuda(w.conv_w), cuda(w.cu_seqlens), cpool, cuda(slots),
                                cuda(w.has_initial_state))
    q, k, v = qkv_views(y, d)
    g, beta = gdn().gdn_gating(cuda(w.a), cuda(w.b), cuda(w.A_log), cuda(w.dt_bias))
    o = gdn().gdn_prefill_chunked(q, k, v, g, beta, cuda(w.cu_seqlens), spool, cuda(none),
                                  cuda(slots), w.scale, chunk=w.chunk, workspace=workspace)
    torch.cuda.synchronize()
    status_clean()
    # every sequence, three heads each (both V heads of some QK heads, and
    # the first and last head)
    picks = [(s, h) for s in range(w.n_seqs) for h in sorted({(3 * s) % 32, 16 + s, 31 - s})]
    import concurrent.futures as cf
    with cf.ThreadPoolExecutor(8) as ex:
        refs = list(ex.map(lambda p: _oracle_chain_from_x(w, *p), picks))
    for (seq, h), (o_ref, S_ref) in zip(picks, refs):
        s, e = int(w.cu_seqlens[seq]), int(w.cu_seqlens[seq + 1])
        assert_close(o[s:e, h], o_ref, TOL[torch.bfloat16], f"o seq {seq} head {h}")
        assert_close(spool[int(slots[seq]), h], S_ref, TOL[torch.bfloat16], f"S seq {seq} head {h}")


def test_long_context_sampled_heads_and_split():
    """T = 65536, nonzero initial state: two heads against the oracle, and
    split-at-32768-and-carry against the single pass on every head."""
    w = workloads.long_context()
    d = w.dims
    q, k, v = cuda(w.q), cuda(w.k), cuda(w.v)
    g, beta = gdn().gdn_gating(cuda(w.a), cuda(w.b), cuda(w.A_log), cuda(w.dt_bias))
    pool = cuda(torch.cat([w.state_pool, torch.zeros(1, d.hv, d.dv, d.dk)]))   # slots 0, 1, 2
    i0 = cuda(torch.tensor([0], dtype=torch.int32))
    f1 = cuda(torch.tensor([1], dtype=torch.int32))
    f2 = cuda(torch.tensor([2], dtype=torch.int32))
    T = w.q.shape[0]
    o = gdn().gdn_prefill_chunked(q, k, v, g, beta, cuda(w.cu_seqlens), pool, i0, f1, w.scale)
    half = T // 2
    cu_h = cuda(torch.tensor([0, half], dtype=torch.int32))
    o1 = gdn().gdn_prefill_chunked(q[:half], k[:half], v[:half], g[:half], beta[:half], cu_h,
                                   pool, i0, f2, w.scale)
    o2 = gdn().gdn_prefill_chunked(q[half:], k[half:], v[half:], g[half:], beta[half:], cu_h,
                                   pool, f2, f2, w.scale)
    torch.cuda.synchronize()
    status_clean()
    assert_close(torch.cat([o1, o2]), o, TOL[torch.bfloat16], "split o")
    assert_close(pool[2], pool[1], TOL[torch.bfloat16], "split final state")

    g_ref, b_ref = oracle_gating(w.a, w.b, w.A_log, w.dt_bias)
    picks = [0, 29]
    res = oracle.gdn_prefill(to_np(w.q), to_np(w.k), to_np(w.v), g_ref, b_ref,
                             to_np(w.cu_seqlens).astype(np.int64), w.state_pool, [0], [1],
                             w.scale, chains=[(0, h) for h in picks], threads=len(picks))
    o_ref, _, finals = res
    for h in picks:
        assert_close(o[:, h], o_ref[:, h], TOL[torch.bfloat16], f"long o head {h}")
        assert_close(pool[1, h], finals[(0, h)], TOL[torch.bfloat16], f"long S head {h}")


def test_prefill_split_matches_fused_every_head():
    """The two tensor-core paths compute the same recurrence but round
    different intermediates to bf16 (the fused kernel X = S K^T, the split
    path W = T diag(beta Gam r_k) K), so on the full 8-sequence batch they
    agree within a few bf16 ulps of max|o| (each is within the 2e-2 bf16
    tolerance of the oracle; here 1e-2 between them)."""
    w = workloads.prefill()
    d = w.dims
    gen = torch.Generator().manual_seed(77)
    T = int(w.cu_seqlens[-1])
    q = cuda(torch.randn(T, d.hqk, d.dk, generator=gen).bfloat16())
    k = cuda(torch.randn(T, d.hqk, d.dk, generator=gen).bfloat16())
    v = cuda(torch.randn(T, d.hv, d.dv, generator=gen).bfloat16())
    g, beta = gdn().gdn_gating(cuda(w.a), cuda(w.b), cuda(w.A_log), cuda(w.dt_bias))
    n = w.cu_seqlens.numel() - 1
    slots = cuda(torch.arange(n, dtype=torch.int32))
    p1 = torch.zeros((n, d.hv, d.dv, d.dk), device=DEV)
    p2 = torch.zeros_like(p1)
    o1 = gdn().gdn_prefill_chunked(q, k, v, g, beta, cuda(w.cu_seqlens), p1, None, slots, w.scale)
    o2 = gdn().gdn_prefill_chunked(q, k, v, g, beta, cuda(w.cu_seqlens), p2, None, slots, w.scale,
                                   workspace=False)
    torch.cuda.synchronize()
    status_clean()
    assert_close(o1, o2, 1e-2, "o split vs fused")
    assert_close(p1, p2, 1e-2, "S split vs fused")


@pytest.fixture(scope="module")
def long_low_decay():
    """T = 65536, one sequence, low decay: A_log ~ U(ln 0.001, ln 0.01), so
    that g is about -0.004 per token and the state carries a few hundred
    tokens of memory across every chunk boundary; initial state ~ N(0, 0.02)."""
    return workloads.long_context(low_decay=True)


def serial_workspace(n_seqs, T, hv):
    """Bytes of the two-kernel path without the chunk-state scan (the header's
    formula): a 1 KiB header, then (ceil(T / 64) + n_seqs) x hv items of
    33 KiB.  A workspace of this size makes a one-sequence call take the
    serial chain."""
    return 1024 + ((T + 63) // 64 + n_seqs) * hv * 33 * 1024


def _long_run(w, pool, init, final, lo, hi, workspace=None):
    q, k, v = cuda(w.q[lo:hi]), cuda(w.k[lo:hi]), cuda(w.v[lo:hi])
    g, beta = gdn().gdn_gating(cuda(w.a[lo:hi]), cuda(w.b[lo:hi]), cuda(w.A_log),
                               cuda(w.dt_bias))
    cu = cuda(torch.tensor([0, hi - lo], dtype=torch.int32))
    if workspace == "serial":
        workspace = torch.empty(serial_workspace(1, hi - lo, w.dims.hv), dtype=torch.uint8,
                                device=DEV)
    return gdn().gdn_prefill_chunked(q, k, v, g, beta, cu, pool,
                                     cuda(torch.tensor([init], dtype=torch.int32)),
                                     cuda(torch.tensor([final], dtype=torch.int32)), w.scale,
                                     workspace=workspace)


def test_long_context_low_decay_carry(long_low_decay):
    """The long-memory carry over 1024 chunks: o and the final state of two
    heads against the oracle's token recurrence, element by element, on the
    chunk-state scan (the default for one long sequence), the serial chain
    and the fused kernel; split at 32768 (scan) and at 32768 + 17 (serial)
    with the state carried through a pool slot against the single pass on
    every head, and against the oracle on the two heads."""
    w = long_low_decay
    d = w.dims
    T = w.q.shape[0]
    ws = gdn().gdn_prefill_workspace_size(1, T, d.hv, d.dk, d.dv, 64)
    assert ws > serial_workspace(1, T, d.hv)          # the default path is the scan
    pool = cuda(torch.cat([w.state_pool, torch.zeros(5, d.hv, d.dv, d.dk)]))  # slots 0 .. 6
    o = _long_run(w, pool, 0, 1, 0, T)
    o_serial = _long_run(w, pool, 0, 4, 0, T, workspace="serial")
    o_fused = _long_run(w, pool, 0, 5, 0, T, workspace=False)
    splits = {}
    for slot, cut, path in ((2, T // 2, None), (3, T // 2 + 17, "serial")):
        oa = _long_run(w, pool, 0, slot, 0, cut, workspace=path)
        ob = _long_run(w, pool, slot, slot, cut, T, workspace=path)
        splits[cut] = (torch.cat([oa, ob]), slot)
    torch.cuda.synchronize()
    status_clean()

    picks = [0, 29]
    g_ref, b_ref = oracle_gating(w.a, w.b, w.A_log, w.dt_bias)
    o_ref, _, finals = oracle.gdn_prefill(
        to_np(w.q), to_np(w.k), to_np(w.v), g_ref, b_ref,
        to_np(w.cu_seqlens).astype(np.int64), w.state_pool, [0], [1], w.scale,
        chains=[(0, h) for h in picks], threads=len(picks))
    tol = TOL[torch.bfloat16]
    for name, oo, slot in (("scan", o, 1), ("serial", o_serial, 4), ("fused", o_fused, 5)):
        for h in picks:
            assert_close(oo[:, h], o_ref[:, h], tol, f"long o head {h} ({name})")
            assert_close(pool[slot, h], finals[(0, h)], tol, f"long S head {h} ({name})")
    assert_close(o, o_serial, tol, "scan vs serial: o")
    assert_close(pool[1], pool[4], tol, "scan vs serial: final state")
    for cut, (o_split, slot) in splits.items():
        assert_close(o_split, o, tol, f"split at {cut}: o")
        assert_close(pool[slot], pool[1], tol, f"split at {cut}: final state")
        for h in picks:
            assert_close(o_split[:, h], o_ref[:, h], tol, f"split at {cut}: o head {h}")
            assert_close(pool[slot, h], finals[(0, h)], tol, f"split at {cut}: S head {h}")


@pytest.mark.parametrize("T,low_decay,init,final", [
    (64 * 70 + 13, True, 0, 0),       # ragged tail, state carried in place
    (64 * 64, True, 1, -1),           # the shortest scanned length, no final slot
    (64 * 201 + 1, False, -1, 2),     # a one-token last chunk, zero initial state
    (64 * 130 + 40, True, 3, 3),
])
def test_chunk_state_scan_small_heads(T, low_decay, init, final):
    """The chunk-state scan of one sequence (split into two segments, the
    second run from zero and from the identity, then combined) against the
    oracle on every head: o and the final state; slots the call must not
    write stay bit-identical.  2 QK / 4 V heads, bf16, dk = dv = 128."""
    hqk, hv = 2, 4
    cu, q, k, v, a, b, A_log, dt_bias, pool = _direct_batch(9000 + T, [T], hqk, hv, 128,
                                                            torch.bfloat16, low_decay, n_slots=4)
    assert gdn().gdn_prefill_workspace_size(1, T, hv, 128, 128, 64) > serial_workspace(1, T, hv)
    ii = torch.tensor([init], dtype=torch.int32)
    fi = torch.tensor([final], dtype=torch.int32)
    pd = cuda(pool)
    g, beta = gdn().gdn_gating(cuda(a), cuda(b), cuda(A_log), cuda(dt_bias))
    o = gdn().gdn_prefill_chunked(cuda(q), cuda(k), cuda(v), g, beta, cuda(cu), pd, cuda(ii),
                                  cuda(fi), 0.0884)
    pd2 = cuda(pool)
    o2 = gdn().gdn_prefill_chunked(cuda(q), cuda(k), cuda(v), g, beta, cuda(cu), pd2, cuda(ii),
                                   cuda(fi), 0.0884,
                                   workspace=torch.empty(serial_workspace(1, T, hv),
                                                         dtype=torch.uint8, device=DEV))
    torch.cuda.synchronize()
    status_clean()
    g_ref, b_ref = oracle_gating(a, b, A_log, dt_bias)
    o_ref, upd, _ = oracle.gdn_prefill(to_np(q), to_np(k), to_np(v), g_ref, b_ref, to_np(cu),
                                       to_np(pool), to_np(ii), to_np(fi), 0.0884)
    tol = TOL[torch.bfloat16]
    assert_close(o, o_ref, tol, "o (scan)")
    assert_close(o2, o_ref, tol, "o (serial)")
    got = pd.cpu()
    for s_ in range(pool.shape[0]):
        for h in range(hv):
            if (s_, h) in upd:
                assert_close(got[s_, h], upd[(s_, h)], tol, f"state {s_},{h}")
            else:
                assert bits_equal(got[s_, h], pool[s_, h]), f"untouched {s_},{h}"
