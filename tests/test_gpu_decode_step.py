"""GPU parity of the fused decode step (conv update + SiLU, gating, L2 norms
and the recurrent update) through the C ABI, on both of its paths (one
kernel without a workspace; the conv / gates kernel and the streaming decode
behind it with one), against the oracle's conv update -> gating -> decode
chain: o and the updated states within the bf16 tolerance, the conv state
pool bit for bit, untouched slots unchanged, at the full decode size (with a
padding row) and at small shapes with one and two V heads per QK head and a
conv bias, and with many more groups than CTAs and padding rows between
them."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_common import DEV, cuda, gdn, oracle_gating, status_clean
from tests.util import TOL, assert_close, bits_equal, to_np
from tests.test_gpu_decode import _state_err, _sub_pool, _untouched

pytestmark = pytest.mark.gpu


PATHS = ["two_kernels", "one_kernel"]


def _check_step(x, conv_w, conv_b, cpool0, a, b, A_log, dt_bias, pool0, idx, hqk, hv, scale,
                path):
    """Run the fused step on copies of the pools and compare with the oracle."""
    cpool = cuda(cpool0)
    pool = cuda(pool0)
    xd = cuda(x)
    workspace = None if path == "two_kernels" else False
    if path == "small_workspace":      # too small: the one-kernel path
        workspace = torch.empty(256, dtype=torch.uint8, device=DEV)
    if path == "unaligned_x":          # rows 8 bytes apart from 16: the one-kernel path
        xd = cuda(torch.nn.functional.pad(x, (0, 4)))[:, :x.shape[1]]
    o = gdn().gdn_decode_step_fused(xd, cuda(conv_w), cpool, cuda(a), cuda(b), cuda(A_log),
                                    cuda(dt_bias), hqk, pool, cuda(idx), scale=scale,
                                    conv_bias=None if conv_b is None else cuda(conv_b),
                                    workspace=workspace)
    torch.cuda.synchronize()
    status_clean()
    live = [int(s) for s in idx if s >= 0]
    y_ref, conv_upd = oracle.conv1d_update(to_np(x), 1, to_np(conv_w),
                                           None if conv_b is None else to_np(conv_b),
                                           to_np(cpool0), to_np(idx).astype(np.int64))
    q_r, k_r, v_r = oracle.split_qkv(y_ref, hqk, hv, 128, 128)
    g_ref, b_ref = oracle_gating(a, b, A_log, dt_bias)
    sub, local = _sub_pool(cuda(pool0), idx)
    o_ref, upd = oracle.gdn_decode(q_r, k_r, v_r, g_ref, b_ref, 1, sub, local, scale=scale)
    assert_close(o, o_ref, TOL[torch.bfloat16], "fused step o")
    dead = (idx < 0)
    assert torch.all(o[dead.to(DEV)] == 0)
    err = _state_err(pool, upd, lambda key: (int(idx[key[0]]), key[1]))
    assert err <= TOL[torch.bfloat16], f"fused step state rel err {err:.3e}"
    assert _untouched(pool, cuda(pool0), set(live))
    got = cpool.cpu()
    for s, st in conv_upd.items():
        assert bits_equal(got[s], torch.from_numpy(st).to(torch.bfloat16)), f"conv slot {s}"
    others = torch.ones(cpool0.shape[0], dtype=torch.bool)
    others[torch.tensor(live, dtype=torch.long)] = False
    assert bits_equal(got[others], cpool0[others])


@pytest.mark.parametrize("path", PATHS)
def test_fused_step_full_size(path):
    """256 sequences x 1 token, 16 QK / 32 V heads, 8192 conv channels, pools
    of 1024 slots; sequence 5 has no slot."""
    w = workloads.decode()
    d = w.dims
    idx = w.slots.clone()
    idx[5] = -1
    _check_step(w.x, w.conv_w, None, w.conv_pool, w.a, w.b, w.A_log, w.dt_bias,
                w.state_pool, idx, d.hqk, d.hv, w.scale, path)


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("hqk,hv", [(2, 4), (4, 4)])
def test_fused_step_small_with_bias(hqk, hv, path):
    g = torch.Generator().manual_seed(91 + hv * hqk)
    n, n_slots = 7, 12
    C = 2 * hqk * 128 + hv * 128
    x = torch.randn(n, C, generator=g).bfloat16()
    conv_w = (torch.rand(C, 4, generator=g) - 0.5).bfloat16()
    conv_b = (torch.randn(C, generator=g) * 0.1).bfloat16()
    cpool0 = torch.randn(n_slots, 3, C, generator=g).bfloat16()
    a = torch.randn(n, hv, generator=g).bfloat16()
    b = torch.randn(n, hv, generator=g).bfloat16()
    A_log, dt_bias = workloads.gating_params(g, hv, False)
    pool0 = torch.randn(n_slots, hv, 128, 128, generator=g) * 0.02
    idx = torch.tensor([3, 0, -1, 11, 7, 1, 5], dtype=torch.int32)
    _check_step(x, conv_w, conv_b, cpool0, a, b, A_log, dt_bias, pool0, idx, hqk, hv,
                128 ** -0.5, path)


@pytest.mark.parametrize("path", PATHS)
def test_fused_step_many_groups_with_padding(path):
    """600 sequences of one QK / two V heads: each persistent CTA loops over
    several groups, with a padding row (no slot) every seventh sequence."""
    g = torch.Generator().manual_seed(4242)
    hqk, hv, n, n_slots = 1, 2, 600, 700
    C = 2 * hqk * 128 + hv * 128
    x = torch.randn(n, C, generator=g).bfloat16()
    conv_w = (torch.rand(C, 4, generator=g) - 0.5).bfloat16()
    cpool0 = torch.randn(n_slots, 3, C, generator=g).bfloat16()
    a = torch.randn(n, hv, generator=g).bfloat16()
    b = torch.randn(n, hv, generator=g).bfloat16()
    A_log, dt_bias = workloads.gating_params(g, hv, False)
    pool0 = torch.randn(n_slots, hv, 128, 128, generator=g) * 0.02
    idx = torch.randperm(n_slots, generator=g)[:n].to(torch.int32)
    idx[::7] = -1
    _check_step(x, conv_w, None, cpool0, a, b, A_log, dt_bias, pool0, idx, hqk, hv,
                128 ** -0.5, path)


@pytest.mark.parametrize("path", ["small_workspace", "unaligned_x"])
def test_fused_step_falls_back_to_one_kernel(path):
    """A workspace below gdn_decode_step_workspace_size, or x rows the
    16-byte vectors cannot take, select the one-kernel path: same results."""
    g = torch.Generator().manual_seed(515)
    hqk, hv, n, n_slots = 2, 4, 9, 16
    C = 2 * hqk * 128 + hv * 128
    x = torch.randn(n, C, generator=g).bfloat16()
    conv_w = (torch.rand(C, 4, generator=g) - 0.5).bfloat16()
    cpool0 = torch.randn(n_slots, 3, C, generator=g).bfloat16()
    a = torch.randn(n, hv, generator=g).bfloat16()
    b = torch.randn(n, hv, generator=g).bfloat16()
    A_log, dt_bias = workloads.gating_params(g, hv, False)
    pool0 = torch.randn(n_slots, hv, 128, 128, generator=g) * 0.02
    idx = torch.randperm(n_slots, generator=g)[:n].to(torch.int32)
    _check_step(x, conv_w, None, cpool0, a, b, A_log, dt_bias, pool0, idx, hqk, hv,
                128 ** -0.5, path)
