"""Shared helpers of the test suite: tolerances and comparisons."""
import numpy as np
import torch

# max |gpu - oracle| / max |oracle|: 1e-4 with fp32 activations, 2e-2 with bf16
# activations and fp32 accumulation (the layer's stated tolerances).
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def to_np(t):
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def rel_err(got, ref):
    got, ref = to_np(got), to_np(ref)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    denom = np.abs(ref).max()
    if denom == 0:
        return float(np.abs(got).max())
    return float(np.abs(got - ref).max() / denom)


def assert_close(got, ref, tol, what=""):
    err = rel_err(got, ref)
    assert err <= tol, f"{what}: rel err {err:.3e} > {tol:.1e}"
    return err


def bits_equal(a: torch.Tensor, b: torch.Tensor) -> bool:
    """Bitwise equality (NaN-safe) of two same-dtype tensors."""
    if a.dtype in (torch.float32,):
        return bool(torch.equal(a.view(torch.int32), b.view(torch.int32)))
    if a.dtype in (torch.bfloat16, torch.float16):
        return bool(torch.equal(a.view(torch.int16), b.view(torch.int16)))
    return bool(torch.equal(a, b))
