"""The decode hot path from a plain C program: tests/csrc/decode_from_c.c uses
only include/minipic.h and the CUDA runtime (device memory, the rotary table,
the workspace size, the decode call and the device error word), and its output
matches the oracle at the fp32 tolerance."""

import glob
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import compare, compare_lse

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_dirs():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    libs = [p for p in [os.path.join(home, "lib64")] + glob.glob(os.path.join(home, "targets", "*", "lib"))
            if os.path.exists(os.path.join(p, "libcudart.so"))]
    return os.path.join(home, "include"), libs[0] if libs else None


def test_decode_from_a_c_program(tmp_path):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    cc = shutil.which("gcc") or shutil.which("cc")
    inc, libdir = _cuda_dirs()
    if cc is None or libdir is None:
        pytest.skip("no C compiler or CUDA runtime library")
    from position_independent_kv_paged_gb300 import _build
    import position_independent_kv_paged_gb300 as mp
    _build.build()
    here = os.path.dirname(mp.library_path())
    exe = str(tmp_path / "decode_from_c")
    subprocess.run([cc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", inc,
                    os.path.join(ROOT, "tests", "csrc", "decode_from_c.c"), "-L", here, "-l:libminipic.so",
                    "-L", libdir, "-lcudart", "-Wl,-rpath," + here, "-Wl,-rpath," + libdir, "-o", exe], check=True)
    w = W.irregular_decode(31, "f32", seq_lens=[0, 1, 40, 300, 700], Hq=8, Hkv=2, d=128)
    dcd = w.decode
    B, mb = dcd.batch, dcd.block_tables.shape[1]
    shape = np.array([B, w.Hq, w.Hkv, w.d, w.kv.num_blocks, mb, w.max_pos], dtype=np.int32)
    files = {"shape.i32": shape, "base.f64": np.array([w.rope_base], dtype=np.float64),
             "k.f32": w.kv.k_pool, "v.f32": w.kv.v_pool, "q.f32": dcd.q,
             "tables.i32": dcd.block_tables, "starts.i32": dcd.block_starts,
             "seq_lens.i32": dcd.seq_lens, "q_pos.i32": dcd.q_pos}
    dtypes = {"i32": np.int32, "f32": np.float32, "f64": np.float64}
    for name, arr in files.items():
        np.ascontiguousarray(arr, dtype=dtypes[name.split(".")[1]]).tofile(str(tmp_path / name))
    run = subprocess.run([exe, str(tmp_path)], capture_output=True, text=True)
    assert run.returncode == 0, run.stderr
    assert "device_error 0" in run.stdout
    out = np.fromfile(str(tmp_path / "out.f32"), dtype=np.float32).reshape(B, w.Hq, w.d)
    lse = np.fromfile(str(tmp_path / "lse.f32"), dtype=np.float32).reshape(B, w.Hq)
    ref, rl = oracle.decode(w)
    compare(out, ref, "f32", "decode from C")
    compare_lse(lse, rl, "f32", "decode from C")
