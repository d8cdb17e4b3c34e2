"""GPU parity of the prefill layer in one call (gdn_prefill_layer: the conv of
the raw q|k|v stream, then the chunked prefill with the gates formed in its
prep kernel from the raw a, b) through the C ABI: against the oracle's layer
(conv -> split -> gating -> gated delta rule) on ragged batches with carried
conv and recurrent states, o and states within the bf16 tolerance and the
conv states bit for bit; and bit for bit against the three calls it replaces
(causal_conv1d_fwd, gdn_gating, gdn_prefill_chunked) on the 8-sequence
serving batch and on one long sequence (the chunk-state scan).  The gated
layer call (gdn_prefill_layer_gated: the gated RMSNorm y written instead of
o) against the oracle's layer + gated RMSNorm, and bit for bit against conv
fwd + gating + gdn_prefill_chunked_gated on its three paths (the norm in the
chain kernel's epilogue, after the scan, and after the plain chain for a z
whose rows a TMA tile cannot read)."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_common import DEV, cuda, gdn, status_clean
from tests.util import TOL, assert_close, bits_equal, to_np

pytestmark = pytest.mark.gpu


def _three_calls(w, cpool, spool, slots, init, final):
    d = w.dims
    y = gdn().causal_conv1d_fwd(cuda(w.x), cuda(w.conv_w), cuda(w.cu_seqlens), cpool, slots,
                                cuda(w.has_initial_state))
    nq = d.hqk * 128
    g, beta = gdn().gdn_gating(cuda(w.a), cuda(w.b), cuda(w.A_log), cuda(w.dt_bias))
    return gdn().gdn_prefill_chunked(y[:, :nq].unflatten(1, (d.hqk, 128)),
                                     y[:, nq:2 * nq].unflatten(1, (d.hqk, 128)),
                                     y[:, 2 * nq:].unflatten(1, (d.hv, 128)), g, beta,
                                     cuda(w.cu_seqlens), spool, init, final, w.scale)


def _layer(w, cpool, spool, slots, init, final):
    return gdn().gdn_prefill_layer(cuda(w.x), cuda(w.conv_w), cpool, slots,
                                   cuda(w.has_initial_state), cuda(w.a), cuda(w.b),
                                   cuda(w.A_log), cuda(w.dt_bias), cuda(w.cu_seqlens),
                                   w.dims.hqk, spool, init, final, scale=w.scale)


@pytest.mark.parametrize("lengths,has", [([70, 1, 130, 64], [1, 1, 1, 1]), ([5, 300], [1, 1]),
                                         ([70, 0, 1, 130, 2], [1, 1, 0, 1, 0])])
def test_prefill_layer_vs_oracle(lengths, has):
    """2 QK / 4 V heads at head_dim 128, ragged lengths (a one-token
    sequence, a chunk-aligned one, an empty one), sequences continuing a
    carried conv state and recurrent state from their slot and others (no
    initial state) starting from zero in both."""
    d = workloads.Dims(hqk=2, hv=4)
    w = workloads.prefill(lengths=lengths, n_slots=len(lengths) + 2, dims=d, low_decay=True)
    w.has_initial_state[:] = torch.tensor(has, dtype=w.has_initial_state.dtype)
    gen = torch.Generator().manual_seed(17)
    pool = torch.randn(len(lengths) + 2, d.hv, 128, 128, generator=gen) * 0.05
    slots = cuda(w.slots)
    init = cuda(torch.where(w.has_initial_state.bool(), w.slots, torch.full_like(w.slots, -1)))
    cpool, spool = cuda(w.conv_pool), cuda(pool)
    o = _layer(w, cpool, spool, slots, init, slots)
    torch.cuda.synchronize()
    status_clean()
    o_ref, conv_upd, upd, _, _, _ = oracle.layer_prefill(
        w.x, w.cu_seqlens, w.conv_w, None, w.conv_pool, w.A_log, w.dt_bias, w.a, w.b, pool,
        w.slots, w.has_initial_state, d.hqk, d.hv, 128, 128, w.scale)
    assert_close(o, o_ref, TOL[torch.bfloat16], "layer o")
    got = spool.cpu()
    for (s, h), st in upd.items():
        assert_close(got[s, h], st, TOL[torch.bfloat16], f"state {s},{h}")
    gotc = cpool.cpu()
    for s, st in conv_upd.items():
        assert bits_equal(gotc[s], torch.from_numpy(st).to(torch.bfloat16)), f"conv slot {s}"


def test_prefill_layer_equals_three_calls_serving_batch():
    """The 8-sequence batch (lengths U{512..8192}): o, the recurrent pool and
    the conv pool bit for bit equal to conv fwd + gating + prefill (the
    prep kernel forms g and beta with the gating kernel's expressions)."""
    w = workloads.prefill()
    d = w.dims
    slots = cuda((w.slots % 64).to(torch.int32))
    none = torch.full_like(slots, -1)
    outs = []
    for fn in (_three_calls, _layer):
        cpool = cuda(w.conv_pool)
        spool = torch.zeros((64, d.hv, 128, 128), device=DEV)
        o = fn(w, cpool, spool, slots, none, slots)
        torch.cuda.synchronize()
        status_clean()
        outs.append((o, spool, cpool))
    for name, a, b in zip(("o", "state pool", "conv pool"), outs[0], outs[1]):
        assert bits_equal(a, b), name


def test_prefill_layer_equals_three_calls_long_sequence():
    """One 8,000-token sequence (the chunk-state scan, its prep kernel fed the
    raw gates) with a carried state: bit for bit equal to the three calls."""
    d = workloads.Dims(hqk=2, hv=4)
    w = workloads.prefill(lengths=[8000], n_slots=2, dims=d, low_decay=True)
    w.has_initial_state[:] = 1
    gen = torch.Generator().manual_seed(23)
    pool = cuda(torch.randn(2, d.hv, 128, 128, generator=gen) * 0.05)
    slots = cuda(w.slots)
    outs = []
    for fn in (_three_calls, _layer):
        cpool, spool = cuda(w.conv_pool), pool.clone()
        o = fn(w, cpool, spool, slots, slots, slots)
        torch.cuda.synchronize()
        status_clean()
        outs.append((o, spool, cpool))
    for name, a, b in zip(("o", "state pool", "conv pool"), outs[0], outs[1]):
        assert bits_equal(a, b), name


def _z(T, hv, pad, seed):
    """z [T, hv, 128] bf16 as a view into rows of hv * 128 + pad elements."""
    gen = torch.Generator().manual_seed(seed)
    zfull = torch.randn(T, hv * 128 + pad, generator=gen).to(torch.bfloat16)
    w = torch.rand(128, generator=gen) + 0.5
    return zfull, w


def _zv(zfull, hv):
    return zfull[:, :hv * 128].unflatten(1, (hv, 128))


def _three_calls_gated(w, cpool, spool, slots, init, final, z, nw):
    d = w.dims
    y = gdn().causal_conv1d_fwd(cuda(w.x), cuda(w.conv_w), cuda(w.cu_seqlens), cpool, slots,
                                cuda(w.has_initial_state))
    nq = d.hqk * 128
    g, beta = gdn().gdn_gating(cuda(w.a), cuda(w.b), cuda(w.A_log), cuda(w.dt_bias))
    return gdn().gdn_prefill_chunked_gated(y[:, :nq].unflatten(1, (d.hqk, 128)),
                                           y[:, nq:2 * nq].unflatten(1, (d.hqk, 128)),
                                           y[:, 2 * nq:].unflatten(1, (d.hv, 128)), g, beta,
                                           cuda(w.cu_seqlens), spool, init, final, w.scale, z,
                                           nw, 1e-6)


def _layer_gated(w, cpool, spool, slots, init, final, z, nw):
    return gdn().gdn_prefill_layer_gated(cuda(w.x), cuda(w.conv_w), cpool, slots,
                                         cuda(w.has_initial_state), cuda(w.a), cuda(w.b),
                                         cuda(w.A_log), cuda(w.dt_bias), cuda(w.cu_seqlens),
                                         w.dims.hqk, spool, init, final, z, nw, 1e-6,
                                         scale=w.scale)


@pytest.mark.parametrize("pad", [64, 4])
def test_prefill_layer_gated_vs_oracle(pad):
    """Ragged lengths with carried conv and recurrent states, 2 QK / 4 V
    heads: y within the bf16 tolerance of the oracle's layer o followed by its
    gated RMSNorm, states as for the plain layer.  A z row stride of
    hv * 128 + 64 lets the chain kernel load z by TMA; + 4 makes the call run
    the plain chain and the norm kernel."""
    lengths = [70, 1, 130, 64]
    d = workloads.Dims(hqk=2, hv=4)
    w = workloads.prefill(lengths=lengths, n_slots=len(lengths) + 2, dims=d, low_decay=True)
    w.has_initial_state[:] = 1
    gen = torch.Generator().manual_seed(19)
    pool = torch.randn(len(lengths) + 2, d.hv, 128, 128, generator=gen) * 0.05
    zfull, nw = _z(w.x.shape[0], d.hv, pad, 29)
    slots = cuda(w.slots)
    cpool, spool = cuda(w.conv_pool), cuda(pool)
    y = _layer_gated(w, cpool, spool, slots, slots, slots, _zv(cuda(zfull), d.hv), cuda(nw))
    torch.cuda.synchronize()
    status_clean()
    o_ref, conv_upd, upd, _, _, _ = oracle.layer_prefill(
        w.x, w.cu_seqlens, w.conv_w, None, w.conv_pool, w.A_log, w.dt_bias, w.a, w.b, pool,
        w.slots, w.has_initial_state, d.hqk, d.hv, 128, 128, w.scale)
    y_ref = oracle.gated_rmsnorm(o_ref, to_np(_zv(zfull, d.hv)), to_np(nw), 1e-6)
    assert_close(y, y_ref, TOL[torch.bfloat16], "layer y")
    got = spool.cpu()
    for (s, h), st in upd.items():
        assert_close(got[s, h], st, TOL[torch.bfloat16], f"state {s},{h}")
    gotc = cpool.cpu()
    for s, st in conv_upd.items():
        assert bits_equal(gotc[s], torch.from_numpy(st).to(torch.bfloat16)), f"conv slot {s}"


@pytest.mark.parametrize("case", ["serving_batch", "long_sequence", "z_not_tma"])
def test_prefill_layer_gated_equals_three_calls(case):
    """y, the recurrent pool and the conv pool bit for bit equal to conv fwd +
    gating + gdn_prefill_chunked_gated: on the 8-sequence batch (the norm in
    the chain epilogue), on one 8,000-token sequence (the chunk-state scan,
    then the norm kernel) and with a z row stride the TMA tile cannot take
    (the plain chain, then the norm kernel)."""
    if case == "long_sequence":
        d = workloads.Dims(hqk=2, hv=4)
        w = workloads.prefill(lengths=[8000], n_slots=2, dims=d, low_decay=True)
        w.has_initial_state[:] = 1
        gen = torch.Generator().manual_seed(31)
        pool = cuda(torch.randn(2, d.hv, 128, 128, generator=gen) * 0.05)
        slots = cuda(w.slots)
        init = final = slots
    else:
        w = workloads.prefill() if case == "serving_batch" else workloads.prefill(
            lengths=[300, 77, 1, 640], n_slots=8, dims=workloads.Dims(hqk=2, hv=4))
        d = w.dims
        slots = cuda((w.slots % 64).to(torch.int32))
        init = torch.full_like(slots, -1)
        final = slots
        pool = torch.zeros((64, d.hv, 128, 128), device=DEV)
    zfull, nw = _z(w.x.shape[0], d.hv, 4 if case == "z_not_tma" else 64, 37)
    z = _zv(cuda(zfull), d.hv)
    outs = []
    for fn in (_three_calls_gated, _layer_gated):
        cpool, spool = cuda(w.conv_pool), pool.clone()
        y = fn(w, cpool, spool, slots, init, final, z, cuda(nw))
        torch.cuda.synchronize()
        status_clean()
        outs.append((y, spool, cpool))
    for name, a, b in zip(("y", "state pool", "conv pool"), outs[0], outs[1]):
        assert bits_equal(a, b), name
