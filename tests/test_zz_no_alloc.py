"""The fixed-scratch prefill entry point (gdn_prefill_chunked_static)
against gdn_prefill_chunked with a caller workspace: the same kernels, so
the outputs and final states must agree bit for bit, on two calls in a row
(a larger problem, then a smaller one that reuses the array), and a problem
past the fixed capacity is refused before anything runs.  Named to run
after the other GPU tests; it also passes alone."""
import numpy as np
import pytest
import torch

from tests.gpu_common import DEV, cuda, gdn, status_clean
from tests.util import bits_equal

pytestmark = pytest.mark.gpu


def _problem(seed, lens, hqk=2, hv=8, n_slots=12):
    gen = torch.Generator().manual_seed(seed)
    T = sum(lens)
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32)
    q = torch.randn(T, hqk, 128, generator=gen).bfloat16()
    k = torch.randn(T, hqk, 128, generator=gen).bfloat16()
    v = torch.randn(T, hv, 128, generator=gen).bfloat16()
    g = -torch.rand(T, hv, generator=gen) * 0.5
    beta = torch.rand(T, hv, generator=gen)
    pool = torch.randn(n_slots, hv, 128, 128, generator=gen) * 0.05
    n = len(lens)
    init = torch.arange(n, dtype=torch.int32)
    init[1] = -1
    final = torch.arange(n, dtype=torch.int32) + n
    return [cuda(t) for t in (q, k, v, g, beta, cu, pool, init, final)]


def _run_both(seed, lens):
    q, k, v, g, beta, cu, pool, init, final = _problem(seed, lens)
    p_ref, p_st = pool.clone(), pool.clone()
    o_ref = gdn().gdn_prefill_chunked(q, k, v, g, beta, cu, p_ref, init, final, 0.0884)
    o_st = gdn().gdn_prefill_chunked_static(q, k, v, g, beta, cu, p_st, init, final, 0.0884)
    torch.cuda.synchronize()
    status_clean()
    assert bits_equal(o_st, o_ref), f"o differs (max {(o_st.float() - o_ref.float()).abs().max()})"
    assert bits_equal(p_st, p_ref), "state pool differs"


def test_static_scratch_matches_workspace_path_twice():
    _run_both(11, [300, 0, 65, 640, 1])        # bound ceil(1006 / 64) + 5 = 21: 168 items
    _run_both(12, [129, 64])                   # fewer items: the array is reused


def test_static_scratch_capacity():
    ws = gdn().gdn_prefill_workspace_size
    cap = gdn().PREFILL_STATIC_SCRATCH_BYTES
    assert ws(5, 1030, 8, 128, 128, 64, gdn().GDN_BF16) <= cap
    lens = [4096, 4096]                        # (128 + 2) x 8 items of 33 KiB = 34 MB: past 16 MiB
    assert ws(2, sum(lens), 8, 128, 128, 64, gdn().GDN_BF16) > cap
    q, k, v, g, beta, cu, pool, init, final = _problem(13, lens)
    before = pool.clone()
    with pytest.raises(gdn().GdnError, match="GDN_ERR_TOO_LARGE"):
        gdn().gdn_prefill_chunked_static(q, k, v, g, beta, cu, pool, init, final, 0.0884)
    torch.cuda.synchronize()
    assert bits_equal(pool, before)
