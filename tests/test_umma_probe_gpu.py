"""The tcgen05 operand layouts, descriptors and TMEM access patterns that the chunked
kernel relies on, checked one MMA chain at a time against a plain matrix product."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

from gpu_util import torch_cuda

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def probe():
    torch_cuda()
    src = os.path.join(HERE, "cuda", "umma_probe.cu")
    lib = os.path.join(HERE, "cuda", "libumma_probe.so")
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
                           "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "-o", lib, src])
    L = ctypes.CDLL(lib)
    L.umma_probe.restype = ctypes.c_int
    L.umma_probe.argtypes = [ctypes.c_int] + [ctypes.c_void_p] * 3 + [ctypes.c_int] * 3 + \
        [ctypes.c_void_p]
    return L


@pytest.mark.parametrize("mode", [0, 1, 2, 3, 4, 6, 8, 10])
@pytest.mark.parametrize("N,K", [(64, 64), (64, 128), (128, 64), (128, 128)])
def test_probe_layouts(probe, mode, N, K):
    torch = torch_cuda()
    g = torch.Generator().manual_seed(mode * 1000 + N + K)
    A = torch.randn(128, K, generator=g).half()
    B = torch.randn(K, N, generator=g).half()
    want = A.double() @ B.double()
    if mode & 8:
        want = -want
    dA, dB = A.cuda(), B.cuda()
    D = torch.full((128, N), float("nan"), device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = probe.umma_probe(mode, dA.data_ptr(), dB.data_ptr(), D.data_ptr(), 128, N, K,
                          st.data_ptr())
    assert rc == 0 and int(st.item()) == 0
    got = D.cpu().double()
    err = (got - want).abs().max().item()
    assert err < 1e-3 * max(1.0, want.abs().max().item()), (mode, N, K, err)
