"""Probe of the tcgen05 building blocks (TMEM A operand, K-major and MN-major SW128 B
operands, shared-memory A operand) against torch matmul, of the exact E4M3 -> bf16
conversion used by the FP8 tensor-core path, and of the bounded mbarrier wait running out."""
import ctypes
import os
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "tc_probe.cu")
SO = os.path.join(HERE, "..", "_build", "libtc_probe.so")


@pytest.fixture(scope="module")
def probe():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    os.makedirs(os.path.dirname(SO), exist_ok=True)
    subprocess.check_call(["/usr/local/cuda/bin/nvcc", "-gencode", "arch=compute_103a,code=sm_103a",
                           "-O2", "-std=c++17", "-Xcompiler", "-fPIC", "-shared", SRC, "-o", SO])
    lib = ctypes.CDLL(SO)
    lib.tc_probe.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + [ctypes.c_void_p]
    lib.e4m3_probe.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.e4m3x4_probe.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int]
    lib.wait_timeout_probe.argtypes = [ctypes.c_void_p]
    return lib


def _run(lib, A, B, K, N, mode):
    D = torch.full((128, N), float("nan"), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert lib.tc_probe(A.data_ptr(), B.data_ptr(), D.data_ptr(), K, N, mode, err.data_ptr()) == 0
    torch.cuda.synchronize()
    assert err.item() == 0
    return D


@pytest.mark.parametrize("mode,K,N", [(0, 64, 16), (0, 64, 32), (0, 128, 64), (0, 128, 256),
                                      (2, 64, 16), (2, 128, 128),
                                      (1, 16, 128), (1, 32, 64), (1, 32, 256), (1, 128, 256),
                                      (3, 32, 128), (3, 32, 256), (3, 64, 128), (3, 64, 256)])
def test_mma_layouts(probe, mode, K, N):
    g = torch.Generator(device="cuda").manual_seed(K * 1000 + N + mode)
    A = torch.randn((128, K), generator=g, device="cuda").to(torch.bfloat16)
    if mode in (1, 3):
        B = torch.randn((K, N), generator=g, device="cuda").to(torch.bfloat16)
        ref = A.float() @ B.float()
    else:
        B = torch.randn((N, K), generator=g, device="cuda").to(torch.bfloat16)
        ref = A.float() @ B.float().t()
    D = _run(probe, A, B, K, N, mode)
    assert torch.allclose(D, ref, atol=1e-3, rtol=1e-4), (D - ref).abs().max().item()


def test_e4m3_to_bf16_exact(probe):
    codes = torch.arange(65536, dtype=torch.int32).to(torch.int16).to("cuda")
    out = torch.empty(65536, dtype=torch.int32, device="cuda")
    assert probe.e4m3_probe(codes.data_ptr(), out.data_ptr(), 65536) == 0
    torch.cuda.synchronize()
    got = out.view(torch.bfloat16).float().view(65536, 2).double() * 2.0 ** 112
    b = codes.view(torch.uint8).view(65536, 2)
    ref = b.view(torch.float8_e4m3fn).double()
    finite = ~torch.isnan(ref)
    assert torch.equal(got[finite], ref[finite])


def test_e4m3x4_to_bf16_exact(probe):
    """The integer E4M3 -> bf16 decode of the FP8 converter: every code in each byte
    position (bytes 0-1 take all 65536 pairs, bytes 2-3 two other sweeps), compared with
    torch's E4M3 decoding; the values must be identical (NaN codes excepted)."""
    i = torch.arange(65536, dtype=torch.int64)
    words = (i & 0xFF) | (((i >> 8) & 0xFF) << 8) | (((i * 37) & 0xFF) << 16) | (((i * 101 + 7) & 0xFF) << 24)
    words = words.to(torch.int32).to("cuda")
    out = torch.empty(65536, 2, dtype=torch.int32, device="cuda")
    assert probe.e4m3x4_probe(words.data_ptr(), out.data_ptr(), 65536) == 0
    torch.cuda.synchronize()
    got = out.view(torch.bfloat16).float().view(65536, 4).double()
    ref = words.view(torch.uint8).view(65536, 4).view(torch.float8_e4m3fn).double()
    finite = ~torch.isnan(ref)
    assert torch.equal(got[finite], ref[finite])


def test_bounded_wait_gives_up_and_reports(probe):
    """A wait nothing satisfies (an mbarrier no thread arrives on): the bounded wait of the
    kernels gives up after its 1 s limit and raises the abort flag, a second waiter sees the
    flag, the kernel finishes, and the context stays usable."""
    out = torch.zeros(3, dtype=torch.int32, device="cuda")
    assert probe.wait_timeout_probe(out.data_ptr()) == 0
    torch.cuda.synchronize()
    gave_up, flag, ms = out.cpu().tolist()
    assert gave_up == 2 and flag == 1
    assert 900 <= ms <= 10000, ms
    assert (torch.ones(4, device="cuda") * 2).sum().item() == 8.0

