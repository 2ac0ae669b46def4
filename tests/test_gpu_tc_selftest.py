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


@pytest.mark.parametrize("N,K,n_off", [(64, 64, 0), (32, 64, 0), (32, 64, 32), (16, 128, 48),
                                       (32, 192, 32)])
def test_m64_result_lanes_and_mn_offset(lib, N, K, n_off):
    """An M=64 MMA leaves result row r in TMEM lane 32*(r//16) + r%16 (16 rows in the
    first half of each 32-lane quadrant, the other lanes untouched), and an MN-major
    operand can start n_off elements into its 128-byte swizzle rows."""
    import torch
    lib.selftest_gemm_m64_probe.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3
    rng = np.random.default_rng(N + K + n_off)
    A, B = _bf16(rng, (64, K)), _bf16(rng, (K, 64))
    dA, dB = A.cuda(), B.cuda()
    dD = torch.full((128, N), 7.0, dtype=torch.float32, device="cuda")
    rc = lib.selftest_gemm_m64_probe(dA.data_ptr(), dB.data_ptr(), dD.data_ptr(), N, K, n_off)
    assert rc == 0, rc
    D = dD.cpu().numpy()
    ref = A.double().numpy() @ B.double().numpy()[:, n_off:n_off + N]
    scale = np.max(np.abs(ref))
    h1 = np.max(np.abs(D[:64] - ref)) / scale
    lanes = np.array([32 * (r // 16) + r % 16 for r in range(64)])
    h2 = np.max(np.abs(D[lanes] - ref)) / scale
    print(f"M=64 N={N} K={K} off={n_off}: rows-in-lanes-0..63 err {h1:.2e}, "
          f"16-rows-per-quadrant err {h2:.2e}")
    others = np.setdiff1d(np.arange(128), lanes)
    assert h2 < 1e-5 and np.all(D[others] == 0.0), (h1, h2)
