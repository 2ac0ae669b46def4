"""GPU pins of the tensor-core building blocks (descriptors, swizzled layouts, TMA).

Builds tests/cuda/tc_selftest.cu (test-only) and checks one tcgen05 MMA tile per
layout combination against a float64 matmul of the same bf16 operands, and that
a 128-byte-swizzled TMA load lands in the layout the kernels assume.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cuda", "tc_selftest.cu")
OUT = os.path.join(HERE, "cuda", "_build", "libtcselftest.so")


@pytest.fixture(scope="module")
def lib():
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    subprocess.run(["nvcc", "-shared", "-Xcompiler", "-fPIC", "-gencode",
                    "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-o", OUT, SRC],
                   check=True)
    lib = ctypes.CDLL(OUT)
    P, I = ctypes.c_void_p, ctypes.c_int
    lib.selftest_gemm_plain.argtypes = [P, P, P, I, I, I, I]
    lib.selftest_gemm_tma.argtypes = [P, P, P, I, I]
    lib.selftest_tma_roundtrip.argtypes = [P, P, I, I]
    return lib


def _bf16(rng, shape):
    import torch
    return torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)


def _ref(a, b):
    return a.double().numpy() @ b.double().numpy()


@pytest.mark.parametrize("a_mn", [0, 1])
@pytest.mark.parametrize("b_mn", [0, 1])
@pytest.mark.parametrize("N,K", [(64, 64), (128, 128), (256, 64), (32, 128), (16, 64),
                                 (192, 192), (64, 16), (128, 256)])
def test_mma_layouts(lib, a_mn, b_mn, N, K):
    import torch
    if b_mn and N > 64 and N % 64:
        pytest.skip("MN-major B wider than one 64-element block must be a multiple of 64")
    rng = np.random.default_rng(N * 1000 + K)
    A, B = _bf16(rng, (128, K)), _bf16(rng, (K, N))
    dA, dB = A.cuda(), B.cuda()
    dD = torch.zeros(128, N, dtype=torch.float32, device="cuda")
    rc = lib.selftest_gemm_plain(dA.data_ptr(), dB.data_ptr(), dD.data_ptr(), N, K, a_mn, b_mn)
    assert rc == 0, rc
    ref = _ref(A, B)
    err = np.max(np.abs(dD.cpu().numpy() - ref)) / np.max(np.abs(ref))
    assert err < 1e-5, err


@pytest.mark.parametrize("R,C", [(64, 64), (128, 128), (192, 64), (64, 256)])
def test_tma_swizzle128_layout(lib, R, C):
    import torch
    rng = np.random.default_rng(R + C)
    src = _bf16(rng, (R, C)).cuda()
    dst = torch.zeros_like(src)
    assert lib.selftest_tma_roundtrip(src.data_ptr(), dst.data_ptr(), R, C) == 0
    assert torch.equal(src, dst)


@pytest.mark.parametrize("N,K", [(64, 64), (128, 128), (256, 64), (192, 192)])
def test_mma_from_tma_operands(lib, N, K):
    import torch
    rng = np.random.default_rng(7 * N + K)
    A, B = _bf16(rng, (128, K)), _bf16(rng, (K, N))
    dA, dB = A.cuda(), B.cuda()   # keep the device copies alive across the call
    dD = torch.zeros(128, N, dtype=torch.float32, device="cuda")
    rc = lib.selftest_gemm_tma(dA.data_ptr(), dB.data_ptr(), dD.data_ptr(), N, K)
    assert rc == 0, rc
    ref = _ref(A, B)
    err = np.max(np.abs(dD.cpu().numpy() - ref)) / np.max(np.abs(ref))
    assert err < 1e-5, err
