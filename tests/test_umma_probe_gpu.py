"""tcgen05 building blocks on the GPU: one CTA computes A.B^T and P.V with the
shared-memory descriptors, instruction descriptor and TMEM moves the prefill
kernel uses; results are compared with float64 products of the same bf16
inputs."""

import ctypes
import os
import subprocess

import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def probe():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    out = os.path.join(ROOT, "_build", "umma_probe.so")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    src = os.path.join(ROOT, "tests", "csrc", "umma_probe.cu")
    inc = os.path.join(ROOT, "position_independent_kv_paged_gb300", "csrc")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-Xcompiler",
                    "-fPIC", "-shared", "-I", inc, "-o", out, src], check=True)
    lib = ctypes.CDLL(out)
    lib.umma_probe.restype = ctypes.c_int
    lib.umma_probe.argtypes = [ctypes.c_void_p] * 8 + [ctypes.c_void_p]
    return torch, lib


def test_tcgen05_products(probe):
    torch, lib = probe
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(0)
    mats = [W.to_bf16_bits(rng.standard_normal((128, 128), dtype=np.float32)) for _ in range(3)]
    Pf = rng.random((128, 128), dtype=np.float32)
    mats.append(W.to_bf16_bits(Pf))
    A, B, V, P = [torch.from_numpy(m.view(np.int16)).to(dev).view(torch.bfloat16) for m in mats]
    S = torch.zeros(128, 128, dtype=torch.float32, device=dev)
    Oss = torch.zeros_like(S)
    Ots = torch.zeros_like(S)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    st = lib.umma_probe(A.data_ptr(), B.data_ptr(), P.data_ptr(), V.data_ptr(), S.data_ptr(), Oss.data_ptr(),
                        Ots.data_ptr(), err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    a, b, v, p = [W.bf16_bits_to_f32(m).astype(np.float64) for m in mats]
    np.testing.assert_allclose(S.cpu().numpy(), a @ b.T, rtol=0, atol=1e-3)
    np.testing.assert_allclose(Oss.cpu().numpy(), p @ v, rtol=0, atol=1e-3)
    np.testing.assert_allclose(Ots.cpu().numpy(), p @ v, rtol=0, atol=1e-3)
