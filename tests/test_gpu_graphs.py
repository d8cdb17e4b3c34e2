"""The C ABI calls are asynchronous on the caller's stream, with no host
synchronisation and no allocation, so a serving loop can capture them in a
CUDA graph: the fused decode step, the two-kernel prefill (with a caller
workspace), the chunk-state scan and the gated prefill, the TMA-staged conv
forward, the one-call prefill layer (plain and gated), the mixed batch with
its decode beside the prefill, and the fused MTP step with its accept copies
are captured with torch.cuda.graph and
replayed (programmatic dependent launches included), and every output and
pool must be bit-identical to an eager run on copies of the same inputs (the
kernels are deterministic)."""
import pytest
import torch

import workloads
from tests.gpu_common import DEV, cuda, gdn, status_clean
from tests.util import bits_equal

pytestmark = pytest.mark.gpu


def _graph(fn):
    """Warm up on a side stream (as torch.cuda.graph wants), capture, replay."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_decode_step_graph_replay():
    """Two replays of the captured step equal two eager steps."""
    w = workloads.decode(pool_device=DEV)
    d = w.dims
    x, a, b = cuda(w.x), cuda(w.a), cuda(w.b)
    conv_w, A_log, dt_bias, slots = cuda(w.conv_w), cuda(w.A_log), cuda(w.dt_bias), cuda(w.slots)
    cpool0, spool0 = cuda(w.conv_pool), w.state_pool

    def run(cpool, spool, o):
        gdn().gdn_decode_step_fused(x, conv_w, cpool, a, b, A_log, dt_bias, d.hqk, spool, slots,
                                    scale=w.scale, o=o)

    ce, se = cpool0.clone(), spool0.clone()
    oe = torch.empty((w.n_seqs, d.hv, d.dv), dtype=x.dtype, device=DEV)
    run(ce, se, oe)
    run(ce, se, oe)
    torch.cuda.synchronize()
    status_clean()

    cg, sg = cpool0.clone(), spool0.clone()
    og = torch.empty_like(oe)
    g = _graph(lambda: run(cg, sg, og))       # warm-up + capture ran the step once
    cg.copy_(cpool0)
    sg.copy_(spool0)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    status_clean()
    assert bits_equal(og, oe)
    assert bits_equal(cg, ce)
    assert bits_equal(sg, se)


def test_prefill_split_graph_replay():
    """The prep + chain prefill with a caller workspace, captured and replayed."""
    w = workloads.prefill()
    d = w.dims
    x = cuda(w.x)
    cu, slots = cuda(w.cu_seqlens), cuda(w.slots)       # conv slots
    y = gdn().causal_conv1d_fwd(x, cuda(w.conv_w), cu, cuda(w.conv_pool), slots,
                                cuda(w.has_initial_state))
    g_, beta = gdn().gdn_gating(cuda(w.a), cuda(w.b), cuda(w.A_log), cuda(w.dt_bias))
    nq = d.hqk * d.dk
    q = y.narrow(1, 0, nq).unflatten(1, (d.hqk, d.dk))
    k = y.narrow(1, nq, nq).unflatten(1, (d.hqk, d.dk))
    v = y.narrow(1, 2 * nq, d.hv * d.dv).unflatten(1, (d.hv, d.dv))
    n_seqs = cu.numel() - 1
    ws = torch.empty(gdn().gdn_prefill_workspace_size(n_seqs, x.shape[0], d.hv, d.dk, d.dv, 64),
                     dtype=torch.uint8, device=DEV)
    # every sequence carries a random initial state in place (slot i)
    sl = torch.arange(n_seqs, dtype=torch.int32, device=DEV)
    gen = torch.Generator(device=DEV).manual_seed(21)
    pool0 = torch.randn(n_seqs, d.hv, d.dv, d.dk, generator=gen, device=DEV) * 0.02

    def run(pool, o):
        gdn().gdn_prefill_chunked(q, k, v, g_, beta, cu, pool, sl, sl, w.scale, o=o, workspace=ws)

    pe = pool0.clone()
    oe = torch.empty((x.shape[0], d.hv, d.dv), dtype=x.dtype, device=DEV)
    run(pe, oe)
    torch.cuda.synchronize()
    status_clean()
    pg = pool0.clone()
    og = torch.empty_like(oe)
    gr = _graph(lambda: run(pg, og))
    pg.copy_(pool0)
    og.zero_()
    gr.replay()
    torch.cuda.synchronize()
    status_clean()
    assert bits_equal(og, oe)
    assert bits_equal(pg, pe)


def test_conv_fwd_graph_replay():
    w = workloads.prefill()
    x, cw, cu, slots, has = (cuda(t) for t in (w.x, w.conv_w, w.cu_seqlens, w.slots,
                                                w.has_initial_state))
    pool0 = cuda(w.conv_pool)
    pe = pool0.clone()
    ye = gdn().causal_conv1d_fwd(x, cw, cu, pe, slots, has)
    torch.cuda.synchronize()
    pg = pool0.clone()
    yg = torch.empty_like(ye)
    gr = _graph(lambda: gdn().causal_conv1d_fwd(x, cw, cu, pg, slots, has, y=yg))
    pg.copy_(pool0)
    yg.zero_()
    gr.replay()
    torch.cuda.synchronize()
    status_clean()
    assert bits_equal(yg, ye)
    assert bits_equal(pg, pe)


def test_scan_and_gated_prefill_graph_replay():
    """The chunk-state scan of one 8,000-token sequence (setup, prep, the
    three-role chain launch, combine, correction) and the gated prefill with
    the norm in the chain's epilogue, captured together and replayed: outputs
    and pools bit-identical to eager runs."""
    gen = torch.Generator().manual_seed(404)
    hqk, hv, T = 2, 4, 8000
    q = cuda(torch.randn(T, hqk, 128, generator=gen).bfloat16())
    k = cuda(torch.randn(T, hqk, 128, generator=gen).bfloat16())
    v = cuda(torch.randn(T, hv, 128, generator=gen).bfloat16())
    g = cuda(-torch.rand(T, hv, generator=gen) * 0.05)
    beta = cuda(torch.rand(T, hv, generator=gen))
    z = cuda(torch.randn(T, hv, 128, generator=gen).bfloat16())
    nw = cuda(torch.rand(128, generator=gen) + 0.5)
    pool0 = cuda(torch.randn(4, hv, 128, 128, generator=gen) * 0.05)
    cu1 = cuda(torch.tensor([0, T], dtype=torch.int32))
    cu2 = cuda(torch.tensor([0, 3000, T], dtype=torch.int32))
    i32 = lambda *x: cuda(torch.tensor(x, dtype=torch.int32))
    s0, s1, s1n, s23 = i32(0), i32(1), i32(1, -1), i32(2, 3)     # made before any capture
    ws1 = torch.empty(gdn().gdn_prefill_workspace_size(1, T, hv, 128, 128, 64), dtype=torch.uint8,
                      device=DEV)
    ws2 = torch.empty(gdn().gdn_prefill_workspace_size(2, T, hv, 128, 128, 64), dtype=torch.uint8,
                      device=DEV)

    def run(pool, o1, o2):
        gdn().gdn_prefill_chunked(q, k, v, g, beta, cu1, pool, s0, s1, 0.0884, o=o1,
                                  workspace=ws1)
        gdn().gdn_prefill_chunked_gated(q, k, v, g, beta, cu2, pool, s1n, s23, 0.0884, z, nw,
                                        1e-6, y=o2, workspace=ws2)

    pe = pool0.clone()
    o1e = torch.empty(T, hv, 128, dtype=torch.bfloat16, device=DEV)
    o2e = torch.empty_like(o1e)
    run(pe, o1e, o2e)
    torch.cuda.synchronize()
    status_clean()

    pg = pool0.clone()
    o1g, o2g = torch.empty_like(o1e), torch.empty_like(o1e)
    gr = _graph(lambda: run(pg, o1g, o2g))
    pg.copy_(pool0)
    gr.replay()
    torch.cuda.synchronize()
    status_clean()
    assert bits_equal(o1g, o1e)
    assert bits_equal(o2g, o2e)
    assert bits_equal(pg, pe)


def test_prefill_layer_graph_replay():
    """gdn_prefill_layer then gdn_prefill_layer_gated on a ragged 4-sequence
    batch (conv into the workspace, chunk offsets, the prep kernel forming
    the gates, the chain kernel with and without the gated epilogue; the
    second call continues the states the first wrote), captured together and
    replayed: o, y, the conv pool and the recurrent pool bit-identical to
    eager runs."""
    d = workloads.Dims(hqk=2, hv=4)
    w = workloads.prefill(lengths=[300, 77, 1, 640], n_slots=6, dims=d, low_decay=True)
    T = w.x.shape[0]
    gen = torch.Generator().manual_seed(405)
    pool0 = cuda(torch.randn(6, d.hv, 128, 128, generator=gen) * 0.05)
    z = cuda(torch.randn(T, d.hv, 128, generator=gen).bfloat16())
    nw = cuda(torch.rand(128, generator=gen) + 0.5)
    x, cw, cu = cuda(w.x), cuda(w.conv_w), cuda(w.cu_seqlens)
    a, b, A_log, dt_bias = cuda(w.a), cuda(w.b), cuda(w.A_log), cuda(w.dt_bias)
    slots, has = cuda(w.slots), cuda(w.has_initial_state)
    none = torch.full_like(slots, -1)
    need = gdn().gdn_prefill_layer_workspace_size(4, T, d.hqk, d.hv)
    raw = torch.empty(need + 1024, dtype=torch.uint8, device=DEV)
    off = (-raw.data_ptr()) % 1024
    ws = raw[off:off + need]

    def run(cpool, pool, o, y):
        gdn().gdn_prefill_layer(x, cw, cpool, slots, has, a, b, A_log, dt_bias, cu, d.hqk, pool,
                                none, slots, scale=w.scale, o=o, workspace=ws)
        gdn().gdn_prefill_layer_gated(x, cw, cpool, slots, has, a, b, A_log, dt_bias, cu, d.hqk,
                                      pool, slots, slots, z, nw, 1e-6, scale=w.scale, y=y,
                                      workspace=ws)

    cpe, pe = cuda(w.conv_pool), pool0.clone()
    oe = torch.empty(T, d.hv, 128, dtype=torch.bfloat16, device=DEV)
    ye = torch.empty_like(oe)
    run(cpe, pe, oe, ye)
    torch.cuda.synchronize()
    status_clean()

    cpg, pg = cuda(w.conv_pool), pool0.clone()
    og, yg = torch.empty_like(oe), torch.empty_like(oe)
    gr = _graph(lambda: run(cpg, pg, og, yg))
    cpg.copy_(cuda(w.conv_pool))
    pg.copy_(pool0)
    gr.replay()
    torch.cuda.synchronize()
    status_clean()
    for name, got, ref in (("o", og, oe), ("y", yg, ye), ("conv pool", cpg, cpe),
                           ("state pool", pg, pe)):
        assert bits_equal(got, ref), name


def test_mixed_batch_and_mtp_step_graph_replay():
    """The mixed batch with the decode beside the prefill's chains (a memset
    of the work counter, the prefill's launches, the streaming decode behind
    the chain kernel) and the fused MTP step with its two accept copies
    (launched behind the MTP kernel), captured and replayed: outputs and
    pools bit-identical to eager runs."""
    w = workloads.mixed(pool_device=DEV)
    d = w.dims
    q, k, v, a, b = (cuda(t) for t in (w.q, w.k, w.v, w.a, w.b))
    cu = cuda(w.cu_seqlens)
    nd = w.extra["n_decode"]
    gg, beta = gdn().gdn_gating(a, b, cuda(w.A_log), cuda(w.dt_bias))
    slots = cuda(w.slots)
    init = torch.where(cuda(w.has_initial_state).bool(), slots, torch.full_like(slots, -1))
    T = q.shape[0]
    need = gdn().gdn_prefill_workspace_size(w.n_seqs - nd, T, d.hv, d.dk, d.dv, 64)
    ws = torch.empty(need + 512, dtype=torch.uint8, device=DEV)

    m = workloads.mtp(n_seqs=16, n_slots=128, pool_device=DEV)
    mx, ma, mb = cuda(m.x), cuda(m.a), cuda(m.b)
    mw, mA, mdt = cuda(m.conv_w), cuda(m.A_log), cuda(m.dt_bias)
    msl, msn = cuda(m.slots), cuda(m.snap)
    acc = cuda(m.snap[torch.arange(m.n_seqs), m.extra["accept"].long()].to(torch.int32))

    def run(pool, o, cpool, spool, mo):
        gdn().gdn_mixed_batch(q, k, v, gg, beta, cu, nd, pool, init, slots, w.scale,
                              decode_in_place=True, o=o, workspace=ws)
        gdn().gdn_mtp_step_fused(mx, 4, mw, cpool, ma, mb, mA, mdt, m.dims.hqk, spool, msl, msn,
                                 scale=m.scale, o=mo)
        gdn().gdn_state_snapshot(spool, acc, msl)
        gdn().gdn_state_snapshot(cpool, acc, msl)

    def fresh():
        return (w.state_pool.clone(), torch.empty((T, d.hv, d.dv), dtype=q.dtype, device=DEV),
                cuda(m.conv_pool), m.state_pool.clone(),
                torch.empty((m.n_seqs * 4, m.dims.hv, m.dims.dv), dtype=mx.dtype, device=DEV))

    eager = fresh()
    run(*eager)
    torch.cuda.synchronize()
    status_clean()
    graphed = fresh()
    gr = _graph(lambda: run(*graphed))
    init_state = fresh()
    for dst, src in zip(graphed, init_state):
        dst.copy_(src)
    gr.replay()
    torch.cuda.synchronize()
    status_clean()
    for name, x_e, x_g in zip(("mixed pool", "mixed o", "conv pool", "state pool", "mtp o"),
                              eager, graphed):
        assert bits_equal(x_g, x_e), name
