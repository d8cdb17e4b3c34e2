"""Helpers shared by the GPU parity tests (CUDA path vs the CPU oracle)."""
import numpy as np
import torch

import oracle
from tests.util import to_np

DEV = "cuda:0"


def gdn():
    import gated_deltanet_linear_10_gb300 as m
    return m


def cuda(t):
    return None if t is None else t.to(DEV)


def status_clean():
    st = gdn().gdn_get_device_status(clear=True)
    assert st == 0, f"device status word {st:#x}"


def oracle_gating(a, b, A_log, dt_bias):
    return oracle.gating(to_np(a), to_np(b), to_np(A_log), to_np(dt_bias))


def qkv_views(y, dims):
    """q, k, v views into a conv output y [T, channels] (row stride = channels)."""
    nq = dims.hqk * dims.dk
    q = y.narrow(1, 0, nq).unflatten(1, (dims.hqk, dims.dk))
    k = y.narrow(1, nq, nq).unflatten(1, (dims.hqk, dims.dk))
    v = y.narrow(1, 2 * nq, dims.hv * dims.dv).unflatten(1, (dims.hv, dims.dv))
    return q, k, v
