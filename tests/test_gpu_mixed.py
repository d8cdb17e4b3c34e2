"""GPU parity of the mixed batch (gdn_mixed_batch: decode rows through the
recurrent decode kernels, the rest through the chunked prefill, one call)
against the oracle's varlen prefill of the same batch, in which a decode row
is a one-token sequence with an initial state: o within the bf16 tolerance,
every final state, untouched slots bit for bit.  Decode rows in place and
into other slots; in the prefill part a zero-initial sequence, a carried
state and a one-token sequence; and the same batch through one
gdn_prefill_chunked call."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_common import cuda, gdn, oracle_gating, status_clean
from tests.test_gpu_prefill import _direct_batch
from tests.util import TOL, assert_close, bits_equal, to_np

pytestmark = pytest.mark.gpu

N_DEC = 20
PRE_LENS = [1, 100, 300]


def _batch():
    hqk, hv = 2, 4
    lens = [1] * N_DEC + PRE_LENS
    n = len(lens)
    n_slots = 2 * n + 4
    cu, q, k, v, a, b, A_log, dt_bias, pool = _direct_batch(909, lens, hqk, hv, 128,
                                                            torch.bfloat16, False, n_slots)
    perm = torch.randperm(n_slots, generator=torch.Generator().manual_seed(5)).to(torch.int32)
    init = perm[:n].clone()                  # slots perm[n:2n] are the "other" final slots
    init[N_DEC + 0] = perm[2 * n]            # the one-token prefill sequence carries a state
    init[N_DEC + 1] = -1                     # a fresh prompt
    return cu, q, k, v, a, b, A_log, dt_bias, pool, init, perm


def _oracle(cu, q, k, v, a, b, A_log, dt_bias, pool, init, final):
    g_ref, b_ref = oracle_gating(a, b, A_log, dt_bias)
    return oracle.gdn_prefill(to_np(q), to_np(k), to_np(v), g_ref, b_ref, to_np(cu), to_np(pool),
                              to_np(init), to_np(final), 0.125)


def _check(o, pd, pool, o_ref, upd):
    assert_close(o, o_ref, TOL[torch.bfloat16], "mixed o")
    got = pd.cpu()
    for s in range(pool.shape[0]):
        for h in range(pool.shape[1]):
            if (s, h) in upd:
                assert_close(got[s, h], upd[(s, h)], TOL[torch.bfloat16], f"state {s},{h}")
            else:
                assert bits_equal(got[s, h], pool[s, h]), f"untouched {s},{h}"


@pytest.mark.parametrize("in_place,path", [(True, "beside"), (True, "serial"), (False, "serial")],
                         ids=["in_place_beside", "in_place_serial", "to_other_slots"])
def test_mixed_batch(in_place, path):
    """In place with the default workspace the decode runs beside the
    prefill's chains (a work counter past the prefill's part); with a
    workspace of exactly the prefill's size the halves run one after the
    other."""
    cu, q, k, v, a, b, A_log, dt_bias, pool, init, perm = _batch()
    n = len(init)
    final = perm[n:2 * n].clone()            # prompts: from their initial slot (or zero)
    final[3] = -1                            # a decode row whose state is dropped
    pd = cuda(pool)
    g, beta = gdn().gdn_gating(cuda(a), cuda(b), cuda(A_log), cuda(dt_bias))
    ws = None
    if path == "serial":
        T = int(cu[-1])
        ws = torch.empty(gdn().gdn_prefill_workspace_size(n - N_DEC, T, 4, 128, 128, 64),
                         dtype=torch.uint8, device="cuda")
    o = gdn().gdn_mixed_batch(cuda(q), cuda(k), cuda(v), g, beta, cuda(cu), N_DEC, pd, cuda(init),
                              cuda(final), 0.125, decode_in_place=in_place, workspace=ws)
    torch.cuda.synchronize()
    status_clean()
    ref_final = final.clone()
    if in_place:                             # decode rows write back into their own slots
        ref_final[:N_DEC] = init[:N_DEC]
    o_ref, upd, _ = _oracle(cu, q, k, v, a, b, A_log, dt_bias, pool, init, ref_final)
    _check(o, pd, pool, o_ref, upd)
    # the same batch through one chunked-prefill call
    p2 = cuda(pool)
    o2 = gdn().gdn_prefill_chunked(cuda(q), cuda(k), cuda(v), g, beta, cuda(cu), p2, cuda(init),
                                   cuda(ref_final), 0.125)
    torch.cuda.synchronize()
    status_clean()
    _check(o2, p2, pool, o_ref, upd)


def test_mixed_batch_all_decode_and_all_prefill():
    """n_decode = n_seqs (no prefill launch) and n_decode = 0 (prefill only)."""
    cu, q, k, v, a, b, A_log, dt_bias, pool, init, perm = _batch()
    n = len(init)
    final = perm[n:2 * n].clone()
    g, beta = gdn().gdn_gating(cuda(a), cuda(b), cuda(A_log), cuda(dt_bias))
    # all decode: the first N_DEC rows as a batch of their own
    cu_d = cu[:N_DEC + 1].clone()
    pd = cuda(pool)
    o = gdn().gdn_mixed_batch(cuda(q[:N_DEC]), cuda(k[:N_DEC]), cuda(v[:N_DEC]), g[:N_DEC],
                              beta[:N_DEC], cuda(cu_d), N_DEC, pd, cuda(init[:N_DEC]),
                              cuda(final[:N_DEC]), 0.125, decode_in_place=False)
    torch.cuda.synchronize()
    status_clean()
    o_ref, upd, _ = _oracle(cu_d, q[:N_DEC], k[:N_DEC], v[:N_DEC], a[:N_DEC], b[:N_DEC], A_log,
                            dt_bias, pool, init[:N_DEC], final[:N_DEC])
    _check(o, pd, pool, o_ref, upd)
    # all prefill
    pd = cuda(pool)
    o = gdn().gdn_mixed_batch(cuda(q), cuda(k), cuda(v), g, beta, cuda(cu), 0, pd, cuda(init),
                              cuda(final), 0.125)
    torch.cuda.synchronize()
    status_clean()
    o_ref, upd, _ = _oracle(cu, q, k, v, a, b, A_log, dt_bias, pool, init, final)
    _check(o, pd, pool, o_ref, upd)


def test_mixed_batch_reports_a_broken_decode_row_layout():
    """Decode rows must be one token each at rows 0 .. n_decode-1; a batch
    whose cu_seqlens breaks that still runs but sets GDN_DEVSTAT_BAD_SEQLEN."""
    cu, q, k, v, a, b, A_log, dt_bias, pool, init, perm = _batch()
    n = len(init)
    final = perm[n:2 * n].clone()
    bad = cu.clone()
    bad[1] = 2                                # decode row 0 claims two tokens
    g, beta = gdn().gdn_gating(cuda(a), cuda(b), cuda(A_log), cuda(dt_bias))
    gdn().gdn_mixed_batch(cuda(q), cuda(k), cuda(v), g, beta, cuda(bad), N_DEC, cuda(pool),
                          cuda(init), cuda(final), 0.125, decode_in_place=False)
    torch.cuda.synchronize()
    st = gdn().gdn_get_device_status(clear=True)
    assert st & gdn().DEVSTAT_BAD_SEQLEN, f"status {st:#x}"


def test_mixed_batch_beside_equals_serial_full_size():
    """The serving-step workload (256 decode rows over 16 QK / 32 V heads,
    two 2048-token prompts): the decode beside the prefill's chains, its
    16,384 items handed out by the counter, gives bit for bit the o and the
    pool of the two halves run one after the other (every item processed
    once, by the same arithmetic)."""
    import workloads
    w = workloads.mixed(pool_device="cuda")
    d = w.dims
    q, k, v, a, b = (cuda(t) for t in (w.q, w.k, w.v, w.a, w.b))
    cu = cuda(w.cu_seqlens)
    nd = w.extra["n_decode"]
    g, beta = gdn().gdn_gating(a, b, cuda(w.A_log), cuda(w.dt_bias))
    slots = cuda(w.slots)
    init = torch.where(cuda(w.has_initial_state).bool(), slots, torch.full_like(slots, -1))
    T = q.shape[0]
    need = gdn().gdn_prefill_workspace_size(w.n_seqs - nd, T, d.hv, d.dk, d.dv, 64)
    outs = []
    for ws_bytes in (need + 512, need):
        pool = w.state_pool.clone()
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        o = gdn().gdn_mixed_batch(q, k, v, g, beta, cu, nd, pool, init, slots, w.scale,
                                  decode_in_place=True, workspace=ws)
        torch.cuda.synchronize()
        status_clean()
        outs.append((o, pool))
    assert bits_equal(outs[0][0], outs[1][0]), "o differs between the two paths"
    assert bits_equal(outs[0][1], outs[1][1]), "pool differs between the two paths"
