"""Cost of one tcgen05.mma (M = 128, K = 16) for the shapes the prefill kernel
issues, in SM cycles (run with -s to see the table).  The prefill tile plan
rests on these numbers: below N of about 96 an MMA costs the same time, so a
narrow key tile wastes tensor throughput."""

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
    out = os.path.join(ROOT, "_build", "mma_rate_probe.so")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    src = os.path.join(ROOT, "tests", "csrc", "mma_rate_probe.cu")
    inc = os.path.join(ROOT, "position_independent_kv_paged_gb300", "csrc")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17", "-Xcompiler",
                    "-fPIC", "-shared", "-I", inc, "-o", out, src], check=True)
    lib = ctypes.CDLL(out)
    lib.mma_rate.restype = ctypes.c_int
    lib.mma_rate.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                             ctypes.c_void_p, ctypes.c_void_p]
    return torch, lib


def cycles_per_mma(probe, n, mode, iters=1000):
    torch, lib = probe
    dev = torch.device("cuda:0")
    ctas = torch.cuda.get_device_properties(dev).multi_processor_count
    cyc = torch.zeros(ctas, dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(2):  # the first launch warms up
        assert lib.mma_rate(cyc.data_ptr(), ctas, n, mode, iters, err.data_ptr(),
                            torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return float(cyc.double().mean().item()) / (8 * iters)


def test_mma_cost_by_shape(probe):
    rows = []
    for mode, n in ((0, 64), (0, 96), (0, 128), (0, 256), (1, 128), (1, 256)):
        c = cycles_per_mma(probe, n, mode)
        rows.append((("SS", "TS")[mode], n, c, 2 * 128 * n * 16 / c))
    print("\nform    N   cycles/MMA   FLOP/cycle/SM")
    for form, n, c, f in rows:
        print(f"{form:4s} {n:4d} {c:11.1f} {f:14.0f}")
    cost = {(form, n): c for form, n, c, _ in rows}
    # a wider MMA never costs less time, and a 256-wide one does more work per cycle
    assert cost[("SS", 64)] <= cost[("SS", 128)] * 1.05 <= cost[("SS", 256)] * 1.05
    assert rows[3][3] > rows[1][3]
