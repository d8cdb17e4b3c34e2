"""GPU parity of the gated RMSNorm (y = o / sqrt(mean(o^2) + eps) * w *
SiLU(z)) through the C ABI against the CPU oracle: the standalone kernel
over head sizes, dtypes, a strided z and in place, and the decode kernel
with the norm fused into its output (full decode size, MTP with snapshots,
the one-CTA layout at dv <= 64 and, at dv = 128, the two-CTA layout
followed by the norm kernel in place; a padding row)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_common import DEV, cuda, gdn, oracle_gating, status_clean
from tests.util import TOL, assert_close, bits_equal, to_np
from tests.test_gpu_decode import _sub_pool

pytestmark = pytest.mark.gpu


def _norm_inputs(seed, T, hv, dv, dtype, zpad=24):
    g = torch.Generator().manual_seed(seed)
    o = (torch.randn(T, hv, dv, generator=g) * 2.0).to(dtype)
    zbig = torch.randn(T, hv * dv + zpad, generator=g).to(dtype)        # z: a strided view
    w = torch.rand(dv, generator=g) + 0.5
    return o, zbig, w


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dv", [16, 64, 128, 256])
def test_standalone_gated_rmsnorm(dtype, dv):
    T, hv = 37, 4        # 16-byte aligned z rows: the bulk-staged kernel
    o, zbig, w = _norm_inputs(dv, T, hv, dv, dtype)
    z = zbig[:, 8:8 + hv * dv].unflatten(1, (hv, dv))
    y = gdn().gdn_gated_rmsnorm(cuda(o), cuda(zbig)[:, 8:8 + hv * dv].unflatten(1, (hv, dv)), cuda(w))
    od = cuda(o)
    yi = gdn().gdn_gated_rmsnorm(od, cuda(zbig)[:, 8:8 + hv * dv].unflatten(1, (hv, dv)), cuda(w), y=od)
    torch.cuda.synchronize()
    ref = oracle.gated_rmsnorm(to_np(o), to_np(z), to_np(w))
    assert_close(y, ref, TOL[dtype], "y")
    assert bits_equal(yi, y)                    # in place gives the same bits


@pytest.mark.parametrize("dtype,hv,dv,off", [(torch.bfloat16, 4, 128, 4),
                                             (torch.bfloat16, 4, 16, 4),
                                             (torch.float32, 32, 256, 8)])
def test_standalone_gated_rmsnorm_register_path(dtype, hv, dv, off):
    """Shapes the bulk-staged kernel leaves to the register kernel: a z view
    8 bytes off a 16-byte boundary (bf16), or tokens larger than half a
    stage (fp32, 32 heads of 256)."""
    T = 29
    o, zbig, w = _norm_inputs(dv + off, T, hv, dv, dtype)
    z = zbig[:, off:off + hv * dv].unflatten(1, (hv, dv))
    y = gdn().gdn_gated_rmsnorm(cuda(o), cuda(zbig)[:, off:off + hv * dv].unflatten(1, (hv, dv)),
                                cuda(w))
    torch.cuda.synchronize()
    ref = oracle.gated_rmsnorm(to_np(o), to_np(z), to_np(w))
    assert_close(y, ref, TOL[dtype], "y")


def _decode_case(dtype, n, tps, hqk, hv, d, seed):
    g = torch.Generator().manual_seed(seed)
    T = n * tps
    q = torch.randn(T, hqk, d, generator=g).to(dtype)
    k = torch.randn(T, hqk, d, generator=g).to(dtype)
    v = torch.randn(T, hv, d, generator=g).to(dtype)
    a = torch.randn(T, hv, generator=g).to(dtype)
    b = torch.randn(T, hv, generator=g).to(dtype)
    A_log, dt_bias = workloads.gating_params(g, hv, False)
    z = torch.randn(T, hv, d, generator=g).to(dtype)
    w = torch.rand(d, generator=g) + 0.5
    pool = torch.randn(n * (tps + 1) + 2, hv, d, d, generator=g) * 0.02
    return q, k, v, a, b, A_log, dt_bias, z, w, pool


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("tps", [1, 4])
def test_decode_gated_small(d, tps):
    """d = 64: one CTA per state, the norm in its epilogue; d = 128: two
    CTAs per state, then the norm kernel in place.  tps = 4 writes per-token snapshots.  Sequence 1 has no slot."""
    dtype = torch.bfloat16
    n, hqk, hv = 6, 2, 4
    q, k, v, a, b, A_log, dt_bias, z, w, pool = _decode_case(dtype, n, tps, hqk, hv, d, 31 * d + tps)
    idx = torch.arange(n, dtype=torch.int32)
    idx[1] = -1
    snap = (torch.arange(n * tps, dtype=torch.int32) + n).view(n, tps) if tps > 1 else None
    g_, beta = gdn().gdn_gating(cuda(a), cuda(b), cuda(A_log), cuda(dt_bias))
    p1, p2 = cuda(pool), cuda(pool)
    y = gdn().gdn_decode_recurrent_gated(cuda(q), cuda(k), cuda(v), g_, beta, tps, p1, cuda(idx),
                                         cuda(z), cuda(w), 1e-6,
                                         snap_indices=None if snap is None else cuda(snap))
    o = gdn().gdn_decode_recurrent(cuda(q), cuda(k), cuda(v), g_, beta, tps, p2, cuda(idx),
                                   snap_indices=None if snap is None else cuda(snap))
    torch.cuda.synchronize()
    status_clean()
    assert bits_equal(p1, p2)                    # the state path is the plain decode's
    g_ref, b_ref = oracle_gating(a, b, A_log, dt_bias)
    o_ref, _ = oracle.gdn_decode(to_np(q), to_np(k), to_np(v), g_ref, b_ref, tps, pool.numpy(),
                                 idx.numpy(), None if snap is None else snap.numpy(),
                                 scale=d ** -0.5)
    y_ref = oracle.gated_rmsnorm(o_ref, to_np(z), to_np(w))
    live = (idx >= 0).repeat_interleave(tps)
    assert_close(y[live], y_ref[live.numpy()], TOL[dtype], "gated decode y")
    assert torch.all(y[~live] == 0)


def test_decode_gated_full_size():
    """256 sequences x 1 token, 32 V heads, dk = dv = 128 (the decode step's
    shapes) with the norm fused: against the oracle's decode + norm."""
    w = workloads.decode(pool_device=DEV)
    d = w.dims
    gen = torch.Generator().manual_seed(2024)
    z = torch.randn(w.q.shape[0], d.hv, d.dv, generator=gen).bfloat16()
    nw = torch.rand(d.dv, generator=gen) + 0.5
    before = w.state_pool.clone()
    q, k, v, a, b = (cuda(t) for t in (w.q, w.k, w.v, w.a, w.b))
    g_, beta = gdn().gdn_gating(a, b, cuda(w.A_log), cuda(w.dt_bias))
    y = gdn().gdn_decode_recurrent_gated(q, k, v, g_, beta, 1, w.state_pool, cuda(w.slots),
                                         cuda(z), cuda(nw), 1e-6, scale=w.scale)
    torch.cuda.synchronize()
    status_clean()
    g_ref, b_ref = oracle_gating(w.a, w.b, w.A_log, w.dt_bias)
    sub, local = _sub_pool(before, w.slots)
    o_ref, _ = oracle.gdn_decode(to_np(w.q), to_np(w.k), to_np(w.v), g_ref, b_ref, 1, sub, local,
                                 scale=w.scale)
    assert_close(y, oracle.gated_rmsnorm(o_ref, to_np(z), to_np(nw)), TOL[torch.bfloat16],
                 "gated decode y")
