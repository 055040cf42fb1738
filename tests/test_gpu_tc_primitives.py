"""GPU check of the tcgen05 building blocks (tc.cuh): one CTA computes D = [C +] A B^T for a
128 x K bf16 A and an N x K bf16 B through shared-memory descriptors and a tensor-memory
accumulator.  Products of bf16 values are exact in fp32, so the result must match an fp64
reference to fp32 accumulation rounding."""
import ctypes
import os
import subprocess

import pytest
import torch

from gated_deltanet_cpr_gb300 import build as gbuild

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def lib():
    src = os.path.join(HERE, "cuda", "tc_selftest.cu")
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libtc_selftest.so")
    subprocess.check_call([gbuild.nvcc(), *gbuild.ARCH, *gbuild.NVCC_FLAGS, "-shared", "-o", so, src])
    L = ctypes.CDLL(so)
    L.tc_selftest.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                                      ctypes.c_void_p]
    L.tc_selftest.restype = ctypes.c_int
    L.transpose_selftest.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_void_p]
    L.transpose_selftest.restype = ctypes.c_int
    L.mn_selftest.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 4 + [ctypes.c_void_p] * 2
    L.mn_selftest.restype = ctypes.c_int
    return L


@pytest.fixture(scope="module")
def inv_lib():
    src = os.path.join(HERE, "cuda", "inverse_selftest.cu")
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libinverse_selftest.so")
    subprocess.check_call([gbuild.nvcc(), *gbuild.ARCH, *gbuild.NVCC_FLAGS, "-shared", "-o", so, src])
    L = ctypes.CDLL(so)
    L.inverse_selftest.argtypes = [ctypes.c_void_p] * 4
    L.inverse_selftest.restype = ctypes.c_int
    return L


@pytest.mark.parametrize("N,K,init", [(64, 128, False), (128, 64, False), (128, 128, True),
                                      (16, 16, False), (256, 32, True)])
def test_tcgen05_mma_matches_reference(lib, N, K, init):
    g = torch.Generator().manual_seed(N * 1000 + K)
    A = torch.randn((128, K), generator=g).to(torch.bfloat16)
    B = torch.randn((N, K), generator=g).to(torch.bfloat16)
    C = torch.randn((128, N), generator=g) if init else None
    ref = A.double() @ B.double().T + (C.double() if init else 0.0)
    dA, dB = A.cuda(), B.cuda()
    dC = C.cuda() if init else None
    D = torch.full((128, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.tc_selftest(dA.data_ptr(), dB.data_ptr(), None if dC is None else dC.data_ptr(),
                         D.data_ptr(), N, K, status.data_ptr(),
                         torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "bounded wait gave up"
    err = (D.double().cpu() - ref).abs().max().item() / ref.abs().max().item()
    assert err < 1e-5, err


@pytest.mark.parametrize("R,Ks", [(128, 64), (64, 64), (64, 128), (16, 32), (128, 128)])
def test_transpose_image_is_exact(lib, R, Ks):
    """The shared-memory image transpose (ldmatrix .trans + stmatrix over core matrices) moves
    every bf16 bit pattern to its transposed place."""
    g = torch.Generator().manual_seed(R * 7 + Ks)
    X = torch.randint(0, 1 << 16, (Ks, R), generator=g, dtype=torch.int32).to(torch.int16)
    dX = X.cuda()
    Y = torch.zeros((R, Ks), dtype=torch.int16, device="cuda")
    rc = lib.transpose_selftest(dX.data_ptr(), Y.data_ptr(), R, Ks, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert torch.equal(Y.cpu(), X.T.contiguous())


@pytest.mark.parametrize("seed,scale", [(0, 0.1), (1, 0.5), (4, 0.2), (5, 0.3), (3, 0.02)])
def test_unrolled_inverse_matches_generic_bits(inv_lib, seed, scale):
    """The unrolled C = 64 inverse of the tensor-core pre-passes performs the generic blocked
    inverse's operations in the same order: same bits, and T (I + A) = I to fp32 accuracy."""
    g = torch.Generator().manual_seed(seed)
    A = (torch.randn((64, 64), generator=g) * scale).tril(-1).contiguous()
    dA = A.cuda()
    Tg = torch.full((64, 64), float("nan"), device="cuda")
    Tf = torch.full((64, 64), float("nan"), device="cuda")
    assert inv_lib.inverse_selftest(dA.data_ptr(), Tg.data_ptr(), Tf.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert torch.equal(Tf, Tg)
    T = Tg.double().cpu()
    resid = (T @ (torch.eye(64, dtype=torch.float64) + A.double()) - torch.eye(64, dtype=torch.float64))
    assert resid.abs().max().item() <= 1e-4 * max(1.0, T.abs().max().item())


def _mn_product(lib, A, B, amode, bmode):
    N, K = B.shape
    D = torch.full((128, N), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.mn_selftest(A.data_ptr(), B.data_ptr(), D.data_ptr(), N, K, amode, bmode, status.data_ptr(),
                         torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "bounded wait gave up"
    return D.cpu()


@pytest.mark.parametrize("N,K", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_mn_major_operands_match_k_major_bits(lib, N, K):
    """An operand read MN-major from the image of its transpose (the instruction descriptor's
    transpose bit; leading offset between core matrices along K, stride offset 128 B along M or
    N) gives the product of the K-major operand, bit for bit, and the fp64 reference to fp32
    accumulation rounding."""
    g = torch.Generator().manual_seed(N * 31 + K)
    A = torch.randn((128, K), generator=g).to(torch.bfloat16)
    B = torch.randn((N, K), generator=g).to(torch.bfloat16)
    ref = A.double() @ B.double().T
    dA, dB = A.cuda(), B.cuda()
    base = _mn_product(lib, dA, dB, 0, 0)
    err = (base.double() - ref).abs().max().item() / ref.abs().max().item()
    assert err < 1e-5, err
    for amode, bmode in ((1, 0), (0, 1), (1, 1)):
        assert torch.equal(_mn_product(lib, dA, dB, amode, bmode), base), (amode, bmode)
