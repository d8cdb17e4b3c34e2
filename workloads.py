"""Seeded synthetic inputs for the Gated DeltaNet layer.

This module draws random numbers and nothing else: it holds none of the
layer's arithmetic.  Both the CUDA path (tests, bench, smoke) and the CPU
oracle consume the tensors it returns, so the two always see the same
inputs.  Every tensor is drawn from a ``torch.Generator`` seeded from the
workload's seed (seed 1000 + workload number) in a fixed order, in fp32, and
cast to the workload's I/O dtype.

Shapes are the GDN layer of the Qwen3-Next hybrid model as the lmdeploy
issue "[Feature] Qwen3-Next-80B-A3B Support" lists them (New attention
kernels: QK 16 heads, V 32 heads, head_dim 128), with a width-4 conv over the
q | k | v channel stream (2*16*128 + 32*128 = 8192 channels).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass
class Dims:
    hqk: int = 16
    hv: int = 32
    dk: int = 128
    dv: int = 128
    width: int = 4

    @property
    def channels(self) -> int:
        return 2 * self.hqk * self.dk + self.hv * self.dv


FULL = Dims()
TINY = Dims(hqk=2, hv=4, dk=16, dv=16, width=4)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _normal(gen, shape, std=1.0, dtype=torch.float32):
    return (torch.randn(shape, generator=gen, dtype=torch.float32) * std).to(dtype)


def _uniform(gen, shape, lo, hi, dtype=torch.float32):
    return (torch.rand(shape, generator=gen, dtype=torch.float32) * (hi - lo) + lo).to(dtype)


def gating_params(gen, hv, low_decay=False):
    """A_log ~ U(0, ln 16) and dt_bias ~ N(0, 0.1), fp32.  low_decay draws
    A_log ~ U(ln 0.001, ln 0.01) so that the state is remembered across many
    chunks (used for the carry tests)."""
    if low_decay:
        A_log = _uniform(gen, (hv,), math.log(0.001), math.log(0.01))
    else:
        A_log = _uniform(gen, (hv,), 0.0, math.log(16.0))
    dt_bias = _normal(gen, (hv,), 0.1)
    return A_log, dt_bias


def conv_weight(gen, channels, width, dtype):
    """Depthwise conv taps [channels, width] ~ U(-0.5, 0.5) (the 1/sqrt(width)
    bound of the usual init); no conv bias."""
    return _uniform(gen, (channels, width), -0.5, 0.5, dtype)


@dataclass
class Workload:
    """Inputs of one batch.  Any field may be None when the workload does
    not use it."""
    name: str
    dims: Dims
    dtype: torch.dtype
    chunk: int = 64
    scale: float = 1.0
    # prefill
    cu_seqlens: torch.Tensor | None = None      # [N+1] int32
    # decode / MTP
    n_seqs: int = 0
    tokens_per_seq: int = 1
    x: torch.Tensor | None = None               # [T, channels] raw qkv stream
    q: torch.Tensor | None = None               # [T, hqk, dk] (when drawn directly)
    k: torch.Tensor | None = None
    v: torch.Tensor | None = None               # [T, hv, dv]
    a: torch.Tensor | None = None               # [T, hv]
    b: torch.Tensor | None = None               # [T, hv]
    A_log: torch.Tensor | None = None           # [hv] fp32
    dt_bias: torch.Tensor | None = None         # [hv] fp32
    conv_w: torch.Tensor | None = None          # [channels, width]
    conv_pool: torch.Tensor | None = None       # [slots, width-1, channels]
    state_pool: torch.Tensor | None = None      # [slots, hv, dv, dk] fp32
    slots: torch.Tensor | None = None           # [N] int32: state slot per sequence
    has_initial_state: torch.Tensor | None = None  # [N] uint8
    snap: torch.Tensor | None = None            # [N, tps] int32
    extra: dict = field(default_factory=dict)

    @property
    def n_tokens(self) -> int:
        if self.x is not None:
            return self.x.shape[0]
        return self.v.shape[0]


def pool_normal(n_slots, dims: Dims, std, seed, device="cpu"):
    """fp32 state pool [n_slots, hv, dv, dk] ~ N(0, std^2).  On a CUDA device
    the values come from that device's generator (same seed, different
    stream of numbers from the CPU one)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.empty((n_slots, dims.hv, dims.dv, dims.dk), dtype=torch.float32, device=device)
    out.normal_(0.0, std, generator=g)
    return out


def tiny(seed=1001, T=64, chunk=16, n_slots=4, low_decay=False):
    """1 sequence of T tokens, 2 QK / 4 V heads, head_dim 16, conv width 4
    over 128 channels, fp32, zero initial state, chunk 16."""
    d = TINY
    gen = _gen(seed)
    x = _normal(gen, (T, d.channels))
    a = _normal(gen, (T, d.hv))
    b = _normal(gen, (T, d.hv))
    A_log, dt_bias = gating_params(gen, d.hv, low_decay)
    w = conv_weight(gen, d.channels, d.width, torch.float32)
    return Workload(
        name=f"tiny_fp32_T{T}", dims=d, dtype=torch.float32, chunk=chunk,
        scale=d.dk ** -0.5, cu_seqlens=torch.tensor([0, T], dtype=torch.int32),
        x=x, a=a, b=b, A_log=A_log, dt_bias=dt_bias, conv_w=w,
        conv_pool=torch.zeros((n_slots, d.width - 1, d.channels)),
        state_pool=torch.zeros((n_slots, d.hv, d.dv, d.dk)),
        slots=torch.tensor([1], dtype=torch.int32),
        has_initial_state=torch.tensor([0], dtype=torch.uint8))


def decode(seed=1002, n_seqs=256, n_slots=1024, dims: Dims = FULL, dtype=torch.bfloat16,
           pool_device="cpu"):
    """Recurrent decode step: n_seqs sequences x 1 token, q/k/v/a/b ~ N(0, 1),
    state pool ~ N(0, 0.02), slots = a seeded permutation subset; plus the
    conv update input x ~ N(0, 1) and a bf16 conv-state pool ~ N(0, 1)."""
    d = dims
    gen = _gen(seed)
    perm = torch.randperm(n_slots, generator=gen)
    slots = perm[:n_seqs].to(torch.int32)
    q = _normal(gen, (n_seqs, d.hqk, d.dk), dtype=dtype)
    k = _normal(gen, (n_seqs, d.hqk, d.dk), dtype=dtype)
    v = _normal(gen, (n_seqs, d.hv, d.dv), dtype=dtype)
    a = _normal(gen, (n_seqs, d.hv), dtype=dtype)
    b = _normal(gen, (n_seqs, d.hv), dtype=dtype)
    A_log, dt_bias = gating_params(gen, d.hv)
    x = _normal(gen, (n_seqs, d.channels), dtype=dtype)
    w = conv_weight(gen, d.channels, d.width, dtype)
    conv_pool = _normal(gen, (n_slots, d.width - 1, d.channels), dtype=dtype)
    pool = pool_normal(n_slots, d, 0.02, seed + 7, pool_device)
    return Workload(
        name=f"decode_N{n_seqs}", dims=d, dtype=dtype, scale=d.dk ** -0.5,
        n_seqs=n_seqs, tokens_per_seq=1, x=x, q=q, k=k, v=v, a=a, b=b,
        A_log=A_log, dt_bias=dt_bias, conv_w=w, conv_pool=conv_pool,
        state_pool=pool, slots=slots)


def mtp(seed=1005, n_seqs=128, tps=4, n_slots=1024, dims: Dims = FULL, dtype=torch.bfloat16,
        pool_device="cpu"):
    """MTP speculative decode: n_seqs sequences x tps tokens (row i*tps + t),
    slots and snapshot slots from one seeded permutation (all distinct)."""
    d = dims
    gen = _gen(seed)
    perm = torch.randperm(n_slots, generator=gen)
    slots = perm[:n_seqs].to(torch.int32)
    snap = perm[n_seqs:n_seqs + n_seqs * tps].to(torch.int32).view(n_seqs, tps)
    T = n_seqs * tps
    q = _normal(gen, (T, d.hqk, d.dk), dtype=dtype)
    k = _normal(gen, (T, d.hqk, d.dk), dtype=dtype)
    v = _normal(gen, (T, d.hv, d.dv), dtype=dtype)
    a = _normal(gen, (T, d.hv), dtype=dtype)
    b = _normal(gen, (T, d.hv), dtype=dtype)
    A_log, dt_bias = gating_params(gen, d.hv)
    x = _normal(gen, (T, d.channels), dtype=dtype)
    w = conv_weight(gen, d.channels, d.width, dtype)
    conv_pool = _normal(gen, (n_slots, d.width - 1, d.channels), dtype=dtype)
    accept = torch.randint(0, tps, (n_seqs,), generator=gen).to(torch.int32)
    pool = pool_normal(n_slots, d, 0.02, seed + 7, pool_device)
    return Workload(
        name=f"mtp_N{n_seqs}x{tps}", dims=d, dtype=dtype, scale=d.dk ** -0.5,
        n_seqs=n_seqs, tokens_per_seq=tps, x=x, q=q, k=k, v=v, a=a, b=b,
        A_log=A_log, dt_bias=dt_bias, conv_w=w, conv_pool=conv_pool,
        state_pool=pool, slots=slots, snap=snap, extra={"accept": accept})


def seq_lengths(gen, n, lo, hi):
    """n integer lengths uniform in [lo, hi] inclusive."""
    return torch.randint(lo, hi + 1, (n,), generator=gen)


def prefill(seed=1003, n_seqs=8, lo=512, hi=8192, lengths=None, n_slots=1024,
            dims: Dims = FULL, dtype=torch.bfloat16, chunk=64, low_decay=False):
    """Chunked varlen prefill: raw qkv stream x ~ N(0, 1) for conv, a/b ~ N(0,1),
    zero initial states, final states to seeded distinct slots."""
    d = dims
    gen = _gen(seed)
    if lengths is None:
        lengths = seq_lengths(gen, n_seqs, lo, hi)
    else:
        lengths = torch.as_tensor(lengths, dtype=torch.int64)
        n_seqs = len(lengths)
    cu = torch.zeros(n_seqs + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lengths, 0).to(torch.int32)
    T = int(cu[-1])
    perm = torch.randperm(n_slots, generator=gen)
    slots = perm[:n_seqs].to(torch.int32)
    x = _normal(gen, (T, d.channels), dtype=dtype)
    a = _normal(gen, (T, d.hv), dtype=dtype)
    b = _normal(gen, (T, d.hv), dtype=dtype)
    A_log, dt_bias = gating_params(gen, d.hv, low_decay)
    w = conv_weight(gen, d.channels, d.width, dtype)
    return Workload(
        name=f"prefill_N{n_seqs}_T{T}", dims=d, dtype=dtype, chunk=chunk,
        scale=d.dk ** -0.5, cu_seqlens=cu, n_seqs=n_seqs, x=x, a=a, b=b,
        A_log=A_log, dt_bias=dt_bias, conv_w=w,
        conv_pool=torch.zeros((n_slots, d.width - 1, d.channels), dtype=dtype),
        slots=slots, has_initial_state=torch.zeros(n_seqs, dtype=torch.uint8),
        extra={"lengths": lengths})


def mixed(seed=1006, n_decode=256, prefill_lens=(2048, 2048), n_slots=1024, dims: Dims = FULL,
          dtype=torch.bfloat16, pool_device="cpu"):
    """A serving step's mixed batch: n_decode one-token decode rows first, then
    prompts of prefill_lens tokens; q/k/v/a/b ~ N(0, 1) drawn directly, state
    pool ~ N(0, 0.02); every sequence has its own slot (seeded permutation),
    the decode rows continue their state, the prompts start from zero."""
    d = dims
    gen = _gen(seed)
    lengths = torch.tensor([1] * n_decode + list(prefill_lens), dtype=torch.int64)
    n = len(lengths)
    cu = torch.zeros(n + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lengths, 0).to(torch.int32)
    T = int(cu[-1])
    slots = torch.randperm(n_slots, generator=gen)[:n].to(torch.int32)
    q = _normal(gen, (T, d.hqk, d.dk), dtype=dtype)
    k = _normal(gen, (T, d.hqk, d.dk), dtype=dtype)
    v = _normal(gen, (T, d.hv, d.dv), dtype=dtype)
    a = _normal(gen, (T, d.hv), dtype=dtype)
    b = _normal(gen, (T, d.hv), dtype=dtype)
    A_log, dt_bias = gating_params(gen, d.hv)
    has = torch.zeros(n, dtype=torch.uint8)
    has[:n_decode] = 1
    pool = pool_normal(n_slots, d, 0.02, seed + 7, pool_device)
    return Workload(
        name=f"mixed_D{n_decode}_P{len(prefill_lens)}", dims=d, dtype=dtype, scale=d.dk ** -0.5,
        cu_seqlens=cu, n_seqs=n, q=q, k=k, v=v, a=a, b=b, A_log=A_log, dt_bias=dt_bias,
        state_pool=pool, slots=slots, has_initial_state=has,
        extra={"n_decode": n_decode, "lengths": lengths})


def long_context(seed=1004, T=65536, dims: Dims = FULL, dtype=torch.bfloat16, chunk=64,
                 n_slots=2, low_decay=False, device="cpu"):
    """One sequence of T tokens with q/k/v/a/b ~ N(0, 1) drawn directly (no
    conv), initial state slot 0 ~ N(0, 0.02), final state to slot 1.  On a
    CUDA device the tensors are drawn there, from that device's generator
    (same seed and distributions, a different stream of numbers from the CPU
    one): the fast path for timing runs, which compare with no oracle."""
    d = dims
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)

    def normal(shape, std=1.0):
        return (torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
                * std).to(dtype)

    q = normal((T, d.hqk, d.dk))
    k = normal((T, d.hqk, d.dk))
    v = normal((T, d.hv, d.dv))
    a = normal((T, d.hv))
    b = normal((T, d.hv))
    A_log, dt_bias = gating_params(_gen(seed + 1) if device != "cpu" else gen, d.hv, low_decay)
    pool = torch.zeros((n_slots, d.hv, d.dv, d.dk), device=device)
    pool[0] = (torch.randn((d.hv, d.dv, d.dk), generator=gen, dtype=torch.float32,
                           device=device) * 0.02)
    return Workload(
        name=f"long_T{T}", dims=d, dtype=dtype, chunk=chunk, scale=d.dk ** -0.5,
        cu_seqlens=torch.tensor([0, T], dtype=torch.int32), n_seqs=1, q=q, k=k, v=v,
        a=a, b=b, A_log=A_log, dt_bias=dt_bias, state_pool=pool,
        slots=torch.tensor([1], dtype=torch.int32),
        extra={"init_idx": torch.tensor([0], dtype=torch.int32)})
