"""The C-ABI library builds, loads and exports every declared symbol; host-side
validation rejects bad arguments before any launch (no GPU needed)."""

import ctypes
import os
import re

import pytest

import position_independent_kv_paged_gb300 as mp
from position_independent_kv_paged_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "minipic.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return mp.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(minipic_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("minipic_rope_table", "minipic_attn_decode", "minipic_attn_prefill",
              "minipic_attn_decode_workspace_size", "minipic_status_string", "minipic_device_error"):
        assert n in names


def test_binding_covers_the_entry_points():
    """Every public name of the binding exists, and every call of the header has
    a Python wrapper (the allocation-free decode is a C-only convenience and the
    status strings live in STATUS)."""
    for n in mp.__all__:
        assert hasattr(mp, n), n
    c_only = {"minipic_attn_decode_noalloc", "minipic_status_string", "minipic_prefix_cache_create",
              "minipic_prefix_cache_destroy", "minipic_prefix_cache_assign", "minipic_prefix_cache_release"}
    renamed = {"minipic_attn_decode_workspace_size": "decode_workspace_size",
               "minipic_attn_prefill_workspace_size": "prefill_workspace_size",
               "minipic_rope_tables": "rope_table"}
    for n in declared_functions():
        if n in c_only:
            continue
        assert renamed.get(n, n[len("minipic_"):]) in mp.__all__, n


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(mp.library_path())
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_status_strings(lib):
    assert lib.minipic_status_string(0) == b"ok"
    assert b"invalid" in lib.minipic_status_string(1)
    assert lib.minipic_status_string(99) == b"unknown status"


def _kv(nb=4, hkv=2, bs=16, d=128, k=0x1000, v=0x2000):
    return mp._KV(k, v, nb, hkv, bs, d)


def _decode(B=1, mb=4, q=0x3000, bt=0x4000, st=0x5000, sl=0x6000, qp=0x7000, out=0x8000):
    return mp._Decode(q, bt, st, sl, qp, B, mb, out, None)


def _call_decode(lib, dtype=1, Hq=4, kv=None, rope=None, db=None, ws=None, ws_n=0, rope_ok=True):
    kv = kv or _kv()
    rope = rope or mp._Rope(0x9000, 1024, kv.head_dim, None, 0xC000)
    db = db or _decode()
    return lib.minipic_attn_decode(dtype, Hq, ctypes.byref(kv), ctypes.byref(rope), ctypes.byref(db),
                                   0.0, ws, ws_n, None)


def test_decode_validation_errors(lib):
    # fake (never dereferenced) pointers: every case fails validation before any launch
    assert _call_decode(lib, dtype=7) == 1
    assert _call_decode(lib, Hq=3) == 1                      # Hq % Hkv != 0
    assert _call_decode(lib, kv=_kv(d=96)) == 2              # head_dim unsupported
    assert _call_decode(lib, kv=_kv(bs=32)) == 2             # block size unsupported
    assert _call_decode(lib, Hq=34, kv=_kv(hkv=2)) == 2      # group of 17 > 16
    assert _call_decode(lib, kv=_kv(k=0x1001)) == 1          # misaligned pool
    assert _call_decode(lib, rope=mp._Rope(0x9000, 1024, 64, None, 0xC000)) == 1   # table head_dim mismatch
    assert _call_decode(lib, rope=mp._Rope(0, 1024, 128)) == 1       # null table
    assert _call_decode(lib, rope=mp._Rope(0x9000, 0, 128)) == 1     # empty table
    assert _call_decode(lib, db=_decode(q=0)) == 1                   # null q
    assert _call_decode(lib, db=_decode(mb=0)) == 1                  # no table width
    assert _call_decode(lib, db=_decode(out=0x8004)) == 1            # misaligned out
    assert _call_decode(lib, db=_decode(B=-1)) == 1
    # batch 0 is a no-op
    assert _call_decode(lib, db=_decode(B=0)) == 0


def test_bf16_decode_needs_the_bf16_table(lib):
    # the bf16 (tensor-core) decode reads the bf16 cos | sin | -sin rows; the
    # fp32 decode does not (its checks fail later, on the fake pointers, only
    # for batch > 0)
    for rope in (mp._Rope(0x9000, 1024, 128), mp._Rope(0x9000, 1024, 128, None, 0xC008)):  # missing, misaligned
        assert _call_decode(lib, rope=rope) == 1
        assert _call_decode(lib, rope=rope, db=_decode(B=0)) == 1
        assert _call_decode(lib, dtype=0, rope=rope, db=_decode(B=0)) == 0


def test_rope_table_bf16_validation(lib):
    f = lib.minipic_rope_table_bf16
    assert f(None, 10, 64, 1e4, None) == 1
    assert f(0x1000, 0, 64, 1e4, None) == 1
    assert f(0x1000, 10, 72, 1e4, None) == 1      # rows of 3 d / 2 bf16 must be whole 16-byte chunks
    assert f(0x1000, 10, 64, 0.0, None) == 1
    assert f(0x1008, 10, 64, 1e4, None) == 1


def test_rope_tables_validation(lib):
    f = lib.minipic_rope_tables
    assert f(None, None, None, 10, 64, 1e4, None) == 1          # no table asked for
    assert f(0x1004, None, None, 10, 64, 1e4, None) == 1        # misaligned
    assert f(None, 0x1008, None, 10, 64, 1e4, None) == 1
    assert f(None, None, 0x1000, 10, 72, 1e4, None) == 1        # bf16 rows need head_dim % 16 == 0
    assert f(0x1000, 0x2000, 0x3000, 0, 64, 1e4, None) == 1
    assert f(0x1000, 0x2000, 0x3000, 10, 64, -1.0, None) == 1


def test_rope_table_validation(lib):
    assert lib.minipic_rope_table(None, 10, 64, 1e4, None) == 1
    assert lib.minipic_rope_table(0x1000, 0, 64, 1e4, None) == 1
    assert lib.minipic_rope_table(0x1000, 10, 63, 1e4, None) == 1
    assert lib.minipic_rope_table(0x1000, 10, 64, -1.0, None) == 1
    assert lib.minipic_rope_table(0x1004, 10, 64, 1e4, None) == 1


def test_prefill_rejects_f32(lib):
    kv = _kv()
    rope = mp._Rope(0x9000, 1024, 128)
    pb = mp._Prefill(0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000, 1, 16, 16, 4, 0xA000, None)
    assert lib.minipic_attn_prefill(0, 4, ctypes.byref(kv), ctypes.byref(rope), ctypes.byref(pb),
                                    0.0, None, 0, None) == 2


def test_prefill_needs_the_fp16_table(lib):
    kv = _kv()
    pb = mp._Prefill(0x3000, 0x4000, 0x5000, 0x6000, 0x7000, 0x8000, 1, 16, 16, 4, 0xA000, None)
    for rope in (mp._Rope(0x9000, 1024, 128), mp._Rope(0x9000, 1024, 128, 0xB008)):  # missing, misaligned
        assert lib.minipic_attn_prefill(1, 4, ctypes.byref(kv), ctypes.byref(rope), ctypes.byref(pb),
                                        0.0, None, 0, None) == 1


def test_rope_table_f16_validation(lib):
    f = lib.minipic_rope_table_f16
    assert f(None, 10, 64, 1e4, None) == 1
    assert f(0x1000, 0, 64, 1e4, None) == 1
    assert f(0x1000, 10, 63, 1e4, None) == 1
    assert f(0x1000, 10, 64, 0.0, None) == 1
    assert f(0x1008, 10, 64, 1e4, None) == 1


def test_workspace_size_is_pure_host(lib):
    n = lib.minipic_attn_decode_workspace_size(8, 64, 8, 128, 8192, 16)
    assert n >= 0
    assert lib.minipic_attn_decode_workspace_size(0, 64, 8, 128, 8192, 16) == 0


def test_kv_append_validation(lib):
    KV, App = mp._KV, mp._Append
    f = lib.minipic_kv_append
    kv = KV(None, None, 4, 2, 16, 128)
    empty = App(None, None, None, None, None, 0, 0, 0, 1)
    assert f(1, ctypes.byref(kv), ctypes.byref(empty), None) == 0            # nothing to do
    assert f(7, ctypes.byref(kv), ctypes.byref(empty), None) == 1            # bad dtype
    assert f(1, None, ctypes.byref(empty), None) == 1                        # no pool
    assert f(1, ctypes.byref(KV(None, None, 4, 2, 16, 96)), ctypes.byref(empty), None) == 2  # head_dim 96
    assert f(1, ctypes.byref(KV(None, None, 4, 2, 8, 128)), ctypes.byref(empty), None) == 2  # block size 8
    bad = App(None, None, None, None, None, -1, 0, 0, 1)
    assert f(1, ctypes.byref(kv), ctypes.byref(bad), None) == 1              # negative batch
    nulls = App(None, None, None, None, None, 2, 5, 3, 1)
    assert f(1, ctypes.byref(kv), ctypes.byref(nulls), None) == 1            # missing pointers


def test_kv_swap_validation(lib):
    KV = mp._KV
    for f in (lib.minipic_kv_swap_out, lib.minipic_kv_swap_in):
        kv = KV(None, None, 4, 2, 16, 128)
        assert f(1, ctypes.byref(kv), None, 0, None, None, None) == 0      # nothing to move
        assert f(9, ctypes.byref(kv), None, 0, None, None, None) == 1      # bad dtype
        assert f(1, None, None, 1, None, None, None) == 1                  # no pool
        assert f(1, ctypes.byref(KV(None, None, 4, 2, 16, 80)), None, 1, None, None, None) == 2
        assert f(1, ctypes.byref(kv), None, -1, None, None, None) == 1     # negative count
        assert f(1, ctypes.byref(kv), None, 3, None, None, None) == 1      # missing pointers


def test_plain_c_program_uses_the_host_calls(lib, tmp_path):
    """include/minipic.h compiles as strict C99 and a C program linked against
    libminipic.so gets the block hashes and prefix-cache tables the oracle gives
    (SSEP span shared at two offsets)."""
    import shutil
    import subprocess

    import numpy as np

    import oracle.blockhash as bh

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    libdir = os.path.dirname(mp.library_path())
    exe = str(tmp_path / "abi_from_c")
    subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "csrc", "abi_from_c.c"), "-L", libdir, "-l:libminipic.so",
                    "-Wl,-rpath," + libdir, "-o", exe], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout.splitlines()
    rec = {ln.split()[0]: ln.split()[1:] for ln in out}
    assert rec["status"] == ["invalid", "argument"] and rec["workspace"] == ["1"] and "done" in rec
    ssep, pdep, bs = -7, -9, 4
    p1 = [1, 2, 3, 4, ssep, 11, 12, 13, pdep, 21, 22, 23, 5, 6]
    p2 = [7, 7, 7, 7, 8, 8, 8, 8, ssep, 11, 12, 13, pdep, 31, 32, 33]
    h1 = bh.block_hashes(p1, bs, ssep, pdep, 0x1234)
    h2 = bh.block_hashes(p2, bs, ssep, pdep, 0x1234)
    assert [int(x) for x in rec["hashes1"]] == h1 and [int(x) for x in rec["hashes2"]] == h2
    cache = bh.PrefixCache(16)
    for key, hs in (("tables1", h1), ("tables2", h2)):
        t, s, f = cache.assign(hs, 4, bs)
        want = [f"{int(a)}:{int(b)}:{int(c)}" for a, b, c in zip(t, s, f)]
        assert rec[key] == want, key
    assert h1[1] == h2[2] and rec["tables1"][1].split(":")[0] == rec["tables2"][2].split(":")[0]
    assert np.int64(rec["tables1"][1].split(":")[1]) != np.int64(rec["tables2"][2].split(":")[1])


def test_binding_has_no_cpu_fallback(lib):
    """Every attention entry of the binding refuses host tensors (no CPU path
    exists), and a missing library is an error, not a silent fallback."""
    torch = pytest.importorskip("torch")
    q = torch.zeros(2, 4, 128, dtype=torch.bfloat16)
    pool = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16)
    i32 = torch.zeros(2, 4, dtype=torch.int32)
    v32 = torch.zeros(2, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        mp.attn_decode(q, pool, pool, i32, i32, v32, v32, torch.zeros(16, 128))
    with pytest.raises(ValueError, match="CUDA tensor"):
        mp.attn_prefill(q, torch.zeros(3, dtype=torch.int32), v32, pool, pool, i32, i32, v32,
                        torch.zeros(16, 128), max_q_len=1)
    import importlib
    import subprocess
    import sys
    code = ("import position_independent_kv_paged_gb300 as mp\n"
            "try:\n    mp.load('/nonexistent/libminipic.so')\nexcept mp.MiniPICError as e:\n    print('refused')\n")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True).stdout
    assert "refused" in out
    importlib.import_module("position_independent_kv_paged_gb300")
