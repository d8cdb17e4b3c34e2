"""Failure path of the tensor-core prefill on the GPU, without a fault: the
prep kernel's bounded waits are made to run out (the wait limit shortened to
1 ms and its K|Q loads suppressed, so the barrier they would complete is never
completed), and the kernel must return, report GDN_DEVSTAT_TIMEOUT in the
device status word and leave the context usable: the same call with the
defaults restored then matches the oracle."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_common import cuda, gdn, oracle_gating, status_clean
from tests.util import TOL, assert_close, to_np

pytestmark = pytest.mark.gpu


def _problem(seed=31, lens=(100, 70), hqk=2, hv=4, n_slots=4):
    gen = torch.Generator().manual_seed(seed)
    T = sum(lens)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    q = torch.randn(T, hqk, 128, generator=gen).bfloat16()
    k = torch.randn(T, hqk, 128, generator=gen).bfloat16()
    v = torch.randn(T, hv, 128, generator=gen).bfloat16()
    a = torch.randn(T, hv, generator=gen).bfloat16()
    b = torch.randn(T, hv, generator=gen).bfloat16()
    A_log = torch.rand(hv, generator=gen) * 2.7
    dt_bias = torch.randn(hv, generator=gen) * 0.1
    pool = torch.randn(n_slots, hv, 128, 128, generator=gen) * 0.02
    return cu, q, k, v, a, b, A_log, dt_bias, pool


def test_prep_wait_runs_out_and_the_context_survives():
    cu, q, k, v, a, b, A_log, dt_bias, pool = _problem()
    init = torch.tensor([0, -1], dtype=torch.int32)
    final = torch.tensor([2, 3], dtype=torch.int32)
    g, beta = gdn().gdn_gating(cuda(a), cuda(b), cuda(A_log), cuda(dt_bias))
    status_clean()

    gdn().gdn_debug_set_wait_limit(1_000_000, drop_prep_loads=True)      # 1 ms
    try:
        gdn().gdn_prefill_chunked(cuda(q), cuda(k), cuda(v), g, beta, cuda(cu), cuda(pool),
                                  cuda(init), cuda(final), 0.0884)
        torch.cuda.synchronize()
        st = gdn().gdn_get_device_status(clear=True)
    finally:
        gdn().gdn_debug_set_wait_limit(0, drop_prep_loads=False)
    assert st & gdn().DEVSTAT_TIMEOUT, f"status {st:#x}: the wait did not run out"
    assert st & ~gdn().DEVSTAT_TIMEOUT == 0, f"status {st:#x}"

    # defaults restored: the same call is correct and raises nothing
    pd = cuda(pool)
    o = gdn().gdn_prefill_chunked(cuda(q), cuda(k), cuda(v), g, beta, cuda(cu), pd, cuda(init),
                                  cuda(final), 0.0884)
    torch.cuda.synchronize()
    status_clean()
    g_ref, b_ref = oracle_gating(a, b, A_log, dt_bias)
    o_ref, upd, _ = oracle.gdn_prefill(to_np(q), to_np(k), to_np(v), g_ref, b_ref, to_np(cu),
                                       to_np(pool), to_np(init), to_np(final), 0.0884)
    assert_close(o, o_ref, TOL[torch.bfloat16], "o after the timeout")
    for (s, h), S in upd.items():
        assert_close(pd[s, h], S, TOL[torch.bfloat16], f"state {s},{h}")
