"""The bounded wait behind every pipeline in the library, run out on purpose
without any fault: a kernel waits on an mbarrier phase that nothing completes,
gives up after its limit, reports it in a status word, and the CUDA context
stays usable.  (The library's kernels take the same helper with a 2 s limit
and then set the timeout bit of the device error word.)"""

import ctypes
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def probe():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    out = os.path.join(ROOT, "_build", "wait_probe.so")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    src = os.path.join(ROOT, "tests", "csrc", "wait_probe.cu")
    inc = os.path.join(ROOT, "position_independent_kv_paged_gb300", "csrc")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-Xcompiler",
                    "-fPIC", "-shared", "-I", inc, "-o", out, src], check=True)
    lib = ctypes.CDLL(out)
    lib.wait_probe.restype = ctypes.c_int
    lib.wait_probe.argtypes = [ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_void_p]
    return torch, lib


@pytest.mark.parametrize("limit_ns", [1_000_000, 50_000_000])
def test_wait_that_nothing_ends_gives_up_and_reports(probe, limit_ns):
    torch, lib = probe
    dev = torch.device("cuda:0")
    st = torch.zeros(3, dtype=torch.int64, device=dev)
    assert lib.wait_probe(st.data_ptr(), limit_ns, torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    gave_up, completed, elapsed = (int(x) for x in st.cpu())
    assert gave_up == 2, "the wait on a phase nothing completes must give up"
    assert completed == 1, "the wait on a completed phase must succeed"
    assert limit_ns <= elapsed < limit_ns + 1_000_000_000
    # the context is still usable after the timed-out wait
    x = torch.arange(1024, device=dev, dtype=torch.float32)
    assert float(x.sum().item()) == 1023 * 1024 / 2
