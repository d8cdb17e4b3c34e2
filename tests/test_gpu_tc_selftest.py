"""Self-test of the library's tcgen05 / TMA / TMEM primitives (csrc/tc.cuh):
a one-CTA bf16 GEMM with fp32 accumulation in tensor memory, against a
PyTorch fp32 matmul of the same bf16 values.  Covers K-major and MN-major
shared-memory operands (128-byte swizzle, TMA-loaded) for either side and an
A operand read from tensor memory."""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def selftest_lib():
    out = os.path.join(ROOT, "_build", "libtc_selftest.so")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    csrc = os.path.join(ROOT, "gated_deltanet_linear_10_gb300", "csrc")
    cmd = ["nvcc", "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a",
           "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"),
           "-I", csrc, "-shared", "-o", out, os.path.join(ROOT, "tests", "cuda", "tc_selftest.cu"),
           os.path.join(csrc, "tmap.cu")]
    subprocess.check_call(cmd)
    lib = ctypes.CDLL(out)
    lib.tc_selftest_gemm.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p]
    lib.tc_selftest_gemm.restype = ctypes.c_int
    return lib


@pytest.mark.parametrize("mode", [0, 1, 2, 3])
@pytest.mark.parametrize("N,K", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_tc_gemm(selftest_lib, mode, N, K):
    gen = torch.Generator().manual_seed(mode * 100 + N + K)
    A = torch.randn(128, K, generator=gen).to(torch.bfloat16)
    B = torch.randn(N, K, generator=gen).to(torch.bfloat16)          # D = A @ B^T
    Bdev = B.t().contiguous() if mode == 1 else B                      # mode 1 passes [K][N]
    Adev = A.t().contiguous() if mode == 3 else A                      # mode 3 passes [K][128]
    Ad, Bd = Adev.cuda(), Bdev.cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = selftest_lib.tc_selftest_gemm(Ad.data_ptr(), Bd.data_ptr(), D.data_ptr(), N, K, mode,
                                       err.data_ptr())
    assert rc == 0
    assert int(err.item()) == 0, "bounded wait timed out"
    ref = A.float() @ B.float().t()
    diff = (D.cpu() - ref).abs().max().item()
    assert diff <= 1e-3 * ref.abs().max().item(), f"max diff {diff}"
