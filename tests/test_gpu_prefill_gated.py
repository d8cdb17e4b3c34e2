"""GPU parity of the prefill with the gated RMSNorm written instead of o
(gdn_prefill_chunked_gated) through the C ABI against the CPU oracle: the
oracle's prefill o, then its gated RMSNorm (y = o / sqrt(mean(o^2) + eps) *
w * SiLU(z) per (token, V head) row).  Covers the norm fused into the chain
kernel's output epilogue (bf16, head_dim 128, a workspace), the two-launch
paths (other shapes, the fused prefill kernel, the chunk-state scan), a z
with a free row stride, ragged lengths and the final states."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_common import DEV, cuda, gdn, oracle_gating, qkv_views, status_clean
from tests.util import TOL, assert_close, bits_equal, to_np

pytestmark = pytest.mark.gpu


def _case(seed, lens, hqk, hv, d, dtype, z_pad=64, n_slots=10):
    gen = torch.Generator().manual_seed(seed)
    T = sum(lens)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    q = torch.randn(T, hqk, d, generator=gen).to(dtype)
    k = torch.randn(T, hqk, d, generator=gen).to(dtype)
    v = torch.randn(T, hv, d, generator=gen).to(dtype)
    a = torch.randn(T, hv, generator=gen).to(dtype)
    b = torch.randn(T, hv, generator=gen).to(dtype)
    A_log, dt_bias = workloads.gating_params(gen, hv, low_decay=True)
    pool = torch.randn(n_slots, hv, d, d, generator=gen) * 0.05
    # z as the second half of wider rows: a view with row stride hv * d + z_pad
    zfull = torch.randn(T, hv * d + z_pad, generator=gen).to(dtype)
    w = torch.rand(d, generator=gen) + 0.5
    return cu, q, k, v, a, b, A_log, dt_bias, pool, zfull, w


def _z_view(zfull, hv, d):
    return zfull[:, :hv * d].unflatten(1, (hv, d))


@pytest.mark.parametrize("path", ["fused_epilogue", "no_workspace"])
def test_gated_prefill_head128(path):
    """bf16, dk = dv = 128, chunk 64, ragged lengths up to 10 chunks, nonzero
    initial states, GQA 2 -> 4 heads: with a workspace the norm runs in the
    chain kernel's epilogue, without one it is the fused prefill kernel then
    the norm kernel."""
    lens = [65, 0, 1, 63, 64, 199, 9 * 64 + 13, 2]
    hqk, hv, d = 2, 4, 128
    cu, q, k, v, a, b, A_log, dt_bias, pool, zfull, w = _case(77, lens, hqk, hv, d, torch.bfloat16)
    init = torch.tensor([0, 1, -1, 3, 4, 5, 8, 9], dtype=torch.int32)
    final = torch.tensor([6, 7, 2, 3, -1, 5, 8, -1], dtype=torch.int32)
    pd = cuda(pool)
    zd = cuda(zfull)
    g, beta = gdn().gdn_gating(cuda(a), cuda(b), cuda(A_log), cuda(dt_bias))
    y = gdn().gdn_prefill_chunked_gated(cuda(q), cuda(k), cuda(v), g, beta, cuda(cu), pd,
                                        cuda(init), cuda(final), 0.0884, _z_view(zd, hv, d),
                                        cuda(w), 1e-6,
                                        workspace=None if path == "fused_epilogue" else False)
    torch.cuda.synchronize()
    status_clean()
    g_ref, b_ref = oracle_gating(a, b, A_log, dt_bias)
    o_ref, upd, _ = oracle.gdn_prefill(to_np(q), to_np(k), to_np(v), g_ref, b_ref, to_np(cu),
                                       to_np(pool), to_np(init), to_np(final), 0.0884)
    y_ref = oracle.gated_rmsnorm(o_ref, to_np(_z_view(zfull, hv, d)), to_np(w), 1e-6)
    tol = TOL[torch.bfloat16]
    assert_close(y, y_ref, tol, "y")
    got = pd.cpu()
    for s in range(pool.shape[0]):
        for h in range(hv):
            if (s, h) in upd:
                assert_close(got[s, h], upd[(s, h)], tol, f"state {s},{h}")
            else:
                assert bits_equal(got[s, h], pool[s, h]), f"untouched {s},{h}"


def test_gated_prefill_fused_matches_two_calls_full_layer():
    """The 8-sequence layer (lengths U{512..8192}, conv -> gating -> prefill):
    the gated prefill with the norm in the chain's epilogue against
    gdn_prefill_chunked + gdn_gated_rmsnorm on every head (within 1e-2 of
    max|y|: the fused norm reads the fp32 o, the two calls its bf16
    rounding), and 8 (sequence, head) chains against the oracle."""
    w = workloads.prefill()
    d = w.dims
    gen = torch.Generator().manual_seed(5)
    T = int(w.cu_seqlens[-1])
    z = torch.randn(T, d.hv, d.dv, generator=gen).bfloat16()
    nw = torch.rand(d.dv, generator=gen) + 0.5
    cpool = cuda(w.conv_pool)
    spool = torch.zeros((64, d.hv, d.dv, d.dk), device=DEV)
    slots = (w.slots % 64).to(torch.int32)
    none = torch.full_like(slots, -1)
    y_conv = gdn().causal_conv1d_fwd(cuda(w.x), cuda(w.conv_w), cuda(w.cu_seqlens), cpool,
                                     cuda(slots), cuda(w.has_initial_state))
    q, k, v = qkv_views(y_conv, d)
    g, beta = gdn().gdn_gating(cuda(w.a), cuda(w.b), cuda(w.A_log), cuda(w.dt_bias))
    zd, nwd = cuda(z), cuda(nw)
    y = gdn().gdn_prefill_chunked_gated(q, k, v, g, beta, cuda(w.cu_seqlens), spool, cuda(none),
                                        cuda(slots), w.scale, zd, nwd, 1e-6)
    spool2 = torch.zeros_like(spool)
    o2 = gdn().gdn_prefill_chunked(q, k, v, g, beta, cuda(w.cu_seqlens), spool2, cuda(none),
                                   cuda(slots), w.scale)
    y2 = gdn().gdn_gated_rmsnorm(o2, zd, nwd, 1e-6)
    torch.cuda.synchronize()
    status_clean()
    assert_close(y, y2, 1e-2, "fused vs two calls")
    assert bits_equal(spool, spool2), "final states differ between the gated and plain calls"
    picks = [(s, (5 * s) % 32) for s in range(w.n_seqs)]
    from tests.test_gpu_prefill import _oracle_chain_from_x
    import concurrent.futures as cf
    with cf.ThreadPoolExecutor(8) as ex:
        refs = list(ex.map(lambda p: _oracle_chain_from_x(w, *p), picks))
    for (seq, h), (o_ref, _) in zip(picks, refs):
        s, e = int(w.cu_seqlens[seq]), int(w.cu_seqlens[seq + 1])
        y_ref = oracle.gated_rmsnorm(o_ref, to_np(z[s:e, h]), to_np(nw), 1e-6)
        assert_close(y[s:e, h], y_ref, TOL[torch.bfloat16], f"y seq {seq} head {h}")


@pytest.mark.parametrize("dtype,d,chunk", [(torch.float32, 64, 32), (torch.bfloat16, 32, 16)])
def test_gated_prefill_other_shapes(dtype, d, chunk):
    """Shapes off the tensor-core path: the prefill into y, then the norm in
    place (fp32 at 1e-4, bf16 at 2e-2)."""
    lens = [chunk + 1, 0, 3 * chunk + 7, 1]
    hqk, hv = 2, 4
    cu, q, k, v, a, b, A_log, dt_bias, pool, zfull, w = _case(91 + d, lens, hqk, hv, d, dtype,
                                                              n_slots=6)
    init = torch.tensor([0, -1, 2, 3], dtype=torch.int32)
    final = torch.tensor([4, 5, 2, -1], dtype=torch.int32)
    pd = cuda(pool)
    g, beta = gdn().gdn_gating(cuda(a), cuda(b), cuda(A_log), cuda(dt_bias))
    y = gdn().gdn_prefill_chunked_gated(cuda(q), cuda(k), cuda(v), g, beta, cuda(cu), pd,
                                        cuda(init), cuda(final), 0.3, _z_view(cuda(zfull), hv, d),
                                        cuda(w), 1e-5, chunk=chunk)
    torch.cuda.synchronize()
    status_clean()
    g_ref, b_ref = oracle_gating(a, b, A_log, dt_bias)
    o_ref, upd, _ = oracle.gdn_prefill(to_np(q), to_np(k), to_np(v), g_ref, b_ref, to_np(cu),
                                       to_np(pool), to_np(init), to_np(final), 0.3)
    y_ref = oracle.gated_rmsnorm(o_ref, to_np(_z_view(zfull, hv, d)), to_np(w), 1e-5)
    assert_close(y, y_ref, TOL[dtype], "y")
    for (s, h), S in upd.items():
        assert_close(pd[s, h], S, TOL[dtype], f"state {s},{h}")


def test_gated_prefill_one_long_sequence_scan():
    """One sequence of 8,000 tokens takes the chunk-state scan; the gated
    call is then the scan followed by the norm in place."""
    hqk, hv, d = 2, 4, 128
    cu, q, k, v, a, b, A_log, dt_bias, pool, zfull, w = _case(123, [8000], hqk, hv, d,
                                                              torch.bfloat16, n_slots=2)
    pd = cuda(pool)
    ii, fi = torch.tensor([0], dtype=torch.int32), torch.tensor([1], dtype=torch.int32)
    g, beta = gdn().gdn_gating(cuda(a), cuda(b), cuda(A_log), cuda(dt_bias))
    y = gdn().gdn_prefill_chunked_gated(cuda(q), cuda(k), cuda(v), g, beta, cuda(cu), pd,
                                        cuda(ii), cuda(fi), 0.0884,
                                        _z_view(cuda(zfull), hv, d), cuda(w), 1e-6)
    torch.cuda.synchronize()
    status_clean()
    g_ref, b_ref = oracle_gating(a, b, A_log, dt_bias)
    o_ref, upd, _ = oracle.gdn_prefill(to_np(q), to_np(k), to_np(v), g_ref, b_ref, to_np(cu),
                                       to_np(pool), to_np(ii), to_np(fi), 0.0884)
    y_ref = oracle.gated_rmsnorm(o_ref, to_np(_z_view(zfull, hv, d)), to_np(w), 1e-6)
    assert_close(y, y_ref, TOL[torch.bfloat16], "y")
    for (s, h), S in upd.items():
        assert_close(pd[s, h], S, TOL[torch.bfloat16], f"state {s},{h}")
