"""Pins of the oracle's gated RMSNorm (y = o / sqrt(mean(o^2) + eps) * w *
SiLU(z), the reading taken for the "gated RMSNorm" kernel the Qwen3next
pages name): torch's own rms_norm and silu in fp64, the unit mean square of
a normalised row, scale invariance, and the SiLU identity
SiLU(z) - SiLU(-z) = z (sigma(z) + sigma(-z) = 1)."""
import numpy as np
import torch
import torch.nn.functional as F

import oracle


def _case(seed, n=7, d=128):
    g = torch.Generator().manual_seed(seed)
    o = torch.randn(n, d, generator=g, dtype=torch.float64) * 3.0
    z = torch.randn(n, d, generator=g, dtype=torch.float64) * 2.0
    w = torch.rand(d, generator=g, dtype=torch.float64) + 0.5
    return o, z, w


def test_matches_library_rms_norm_times_silu():
    for d, eps in ((128, 1e-6), (16, 1e-2), (64, 0.0)):
        o, z, w = _case(d, d=d)
        ref = F.rms_norm(o, (d,), w, eps) * F.silu(z)
        y = oracle.gated_rmsnorm(o.numpy(), z.numpy(), w.numpy(), eps)
        np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_unit_mean_square_and_scale_invariance():
    o, z, w = _case(5)
    gate = w.numpy() * F.silu(z).numpy()
    y = oracle.gated_rmsnorm(o.numpy(), z.numpy(), w.numpy(), 0.0)
    np.testing.assert_allclose(np.mean((y / gate) ** 2, axis=-1), 1.0, rtol=1e-12)
    for lam in (1e-3, 7.0, 1e4):
        y2 = oracle.gated_rmsnorm(lam * o.numpy(), z.numpy(), w.numpy(), 0.0)
        np.testing.assert_allclose(y2, y, rtol=1e-12, atol=1e-14)


def test_silu_symmetry_and_zero_gate():
    o, z, w = _case(9)
    on, zn, wn = o.numpy(), z.numpy(), w.numpy()
    ya = oracle.gated_rmsnorm(on, zn, wn, 0.0)
    yb = oracle.gated_rmsnorm(on, -zn, wn, 0.0)
    yz = oracle.gated_rmsnorm(on, np.ones_like(zn) * 40.0, wn, 0.0) / 40.0   # SiLU(40) = 40
    np.testing.assert_allclose(ya - yb, yz * zn, rtol=1e-10, atol=1e-12)
    assert np.all(oracle.gated_rmsnorm(on, np.zeros_like(zn), wn, 1e-6) == 0.0)
    zero = oracle.gated_rmsnorm(np.zeros_like(on), zn, wn, 1e-6)
    assert np.all(np.isfinite(zero)) and np.all(zero == 0.0)
