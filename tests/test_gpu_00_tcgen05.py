"""GPU self-test of the tcgen05 building blocks (shared-memory descriptors with and without
swizzle, the kind::f16 instruction descriptor, tensor-memory loads/stores and the MMA with its
A operand in tensor memory, the MN-major B operand) against torch matmuls."""
import ctypes as C
import os
import subprocess

import pytest

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def lib():
    src = os.path.join(HERE, "gpu_selftest", "umma_selftest.cu")
    out_dir = os.path.join(HERE, "gpu_selftest", "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libumma_selftest.so")
    subprocess.run(["/usr/local/cuda/bin/nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "-Xcompiler", "-fPIC", "-shared", "-o", so, src], check=True)
    l = C.CDLL(so)
    l.umma_selftest.argtypes = [C.c_void_p] * 7
    l.umma_mn_selftest.argtypes = [C.c_void_p] * 4
    l.umma_pair_selftest.argtypes = [C.c_void_p] * 7
    return l


def test_umma_building_blocks(lib):
    g = torch.Generator(device="cpu").manual_seed(0)
    A = torch.randn(128, 144, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(128, 144, generator=g).to(torch.bfloat16).cuda()
    P = torch.rand(128, 128, generator=g).to(torch.bfloat16).cuda()
    Vt = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    S = torch.zeros(128, 128, device="cuda")
    O = torch.zeros(128, 128, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.umma_selftest(A.data_ptr(), B.data_ptr(), P.data_ptr(), Vt.data_ptr(), S.data_ptr(), O.data_ptr(),
                           err.data_ptr())
    assert rc == 0 and err.item() == 0
    S_ref = A.float() @ B.float().T
    O_ref = P.float() @ Vt.float().T
    assert torch.allclose(S, S_ref, rtol=1e-4, atol=1e-3), (S - S_ref).abs().max()
    assert torch.allclose(O, O_ref, rtol=1e-4, atol=1e-3), (O - O_ref).abs().max()


def test_umma_mn_major_b_operand(lib):
    """P V with V stored [key][d] (N contiguous) and read as an MN-major swizzled B operand."""
    g = torch.Generator(device="cpu").manual_seed(1)
    P = torch.rand(128, 128, generator=g).to(torch.bfloat16).cuda()
    V = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    O = torch.zeros(128, 128, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.umma_mn_selftest(P.data_ptr(), V.data_ptr(), O.data_ptr(), err.data_ptr())
    assert rc == 0 and err.item() == 0
    O_ref = P.float() @ V.float()
    assert torch.allclose(O, O_ref, rtol=1e-4, atol=1e-3), (O - O_ref).abs().max()


def test_umma_cta_pair(lib):
    """cta_group::2: M = 256 split over two CTAs, B's N columns split likewise (K-major S, MN-major
    P V with P in each CTA's tensor memory), commits multicast to both CTAs."""
    g = torch.Generator(device="cpu").manual_seed(2)
    A = torch.randn(256, 144, generator=g).to(torch.bfloat16).cuda()
    B = torch.randn(128, 144, generator=g).to(torch.bfloat16).cuda()
    P = torch.rand(256, 128, generator=g).to(torch.bfloat16).cuda()
    V = torch.randn(128, 128, generator=g).to(torch.bfloat16).cuda()
    S = torch.zeros(256, 128, device="cuda")
    O = torch.zeros(256, 128, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.umma_pair_selftest(A.data_ptr(), B.data_ptr(), P.data_ptr(), V.data_ptr(), S.data_ptr(),
                                O.data_ptr(), err.data_ptr())
    assert rc == 0 and err.item() == 0, (rc, err.item())
    S_ref = A.float() @ B.float().T
    O_ref = P.float() @ V.float()
    assert torch.allclose(S, S_ref, rtol=1e-4, atol=1e-3), (S - S_ref).abs().max()
    assert torch.allclose(O, O_ref, rtol=1e-4, atol=1e-3), (O - O_ref).abs().max()
