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
    for fn in (lib.mma_rate, lib.mma_rate2):
        fn.restype = ctypes.c_int
        fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                       ctypes.c_void_p]
    return torch, lib


def cycles_per_mma(probe, n, mode, iters=1000, pair=False):
    torch, lib = probe
    dev = torch.device("cuda:0")
    ctas = torch.cuda.get_device_properties(dev).multi_processor_count
    ctas -= ctas % 2
    cyc = torch.zeros(ctas // 2 if pair else ctas, dtype=torch.int64, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    fn = lib.mma_rate2 if pair else lib.mma_rate
    for _ in range(2):  # the first launch warms up
        assert fn(cyc.data_ptr(), ctas, n, mode, iters, err.data_ptr(), torch.cuda.current_stream().cuda_stream) == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return float(cyc.double().mean().item()) / (8 * iters)


def test_mma_cost_by_shape(probe):
    rows = []
    for mode, n in ((0, 64), (0, 96), (0, 128), (0, 192), (0, 256), (1, 96), (1, 128), (1, 192), (1, 256)):
        c = cycles_per_mma(probe, n, mode)
        rows.append((("SS", "TS")[mode], n, c, 2 * 128 * n * 16 / c))
    print("\nform    N   cycles/MMA   FLOP/cycle/SM")
    for form, n, c, f in rows:
        print(f"{form:4s} {n:4d} {c:11.1f} {f:14.0f}")
    cost = {(form, n): c for form, n, c, _ in rows}
    # a wider MMA never costs less time, and a 256-wide one does more work per cycle
    assert cost[("SS", 64)] <= cost[("SS", 128)] * 1.05 <= cost[("SS", 256)] * 1.05
    assert rows[4][3] > rows[1][3]


def test_pair_mma_cost_by_shape(probe):
    """cta_group::2: M = 256 rows over a CTA pair, N columns (half of B in each
    CTA's shared memory), K = 16; FLOP/cycle is per SM."""
    rows = []
    for mode, n in ((0, 128), (0, 192), (0, 256), (1, 128), (1, 192), (1, 256)):
        c = cycles_per_mma(probe, n, mode, pair=True)
        rows.append((("SS", "TS")[mode], n, c, 256 * n * 16 / c))
    print("\npair form  N   cycles/MMA   FLOP/cycle/SM")
    for form, n, c, f in rows:
        print(f"{form:4s} {n:4d} {c:11.1f} {f:14.0f}")
    assert all(c > 0 for _, _, c, _ in rows)
