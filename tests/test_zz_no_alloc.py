"""The allocation-free decode entry point matches the regular one.

minipic_attn_decode_noalloc serves callers that cannot allocate device memory
at the call (a fixed memory pool, a serving loop where cudaMalloc could
synchronize or fail, a plain C host).  It keeps split-KV partial results in a
fixed device array inside the library.  This test calls it through the C ABI
twice in a row on different inputs (so the second call runs over the first
call's leftover scratch contents) and compares each result with
minipic_attn_decode given a caller workspace.  The calls cover both decode
paths that use split-KV scratch (the bf16 tensor-core kernel, which merges its
splits itself, and the fp32 kernel with its separate merge kernel), and a call
with more split counters than the one before, whose counter region lands on
the earlier call's partial results (the entry point clears it).  The file
sorts last so that a run stopping at the first failure has run every other
test before it.
"""

import ctypes

import numpy as np
import pytest

import workloads as W
from gpu_util import TOL, upload_decode

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from position_independent_kv_paged_gb300 import _build
    _build.build()
    import position_independent_kv_paged_gb300 as mp
    mp.load()
    raw = ctypes.CDLL(mp.library_path())
    fn = raw.minipic_attn_decode_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_int, ctypes.c_int32, ctypes.POINTER(mp._KV), ctypes.POINTER(mp._Rope),
                   ctypes.POINTER(mp._Decode), ctypes.c_float, ctypes.c_void_p]
    return torch, mp, fn, torch.device("cuda:0")


def _noalloc(env, w, t, rope):
    torch, mp, fn, dev = env
    d = w.decode
    out = torch.full_like(t["q"], float("nan"))
    lse = torch.full((d.batch, w.Hq), float("nan"), dtype=torch.float32, device=dev)
    kv = mp._KV(t["k_pool"].data_ptr(), t["v_pool"].data_ptr(), *t["k_pool"].shape)
    rp = mp._Rope(rope.cos_sin.data_ptr(), rope.max_pos, rope.head_dim, None, rope.cos_sin_bf16.data_ptr())
    db = mp._Decode(t["q"].data_ptr(), t["block_tables"].data_ptr(), t["block_starts"].data_ptr(),
                    t["seq_lens"].data_ptr(), t["q_pos"].data_ptr(), d.batch, t["block_tables"].shape[1],
                    out.data_ptr(), lse.data_ptr())
    st = fn(mp.BF16 if w.dtype == "bf16" else mp.F32, w.Hq, ctypes.byref(kv), ctypes.byref(rp),
            ctypes.byref(db), 0.0, torch.cuda.current_stream().cuda_stream)
    assert st == 0, mp.STATUS.get(st)
    return out, lse


def _regular(env, w, t, rope):
    torch, mp, fn, dev = env
    lse = torch.empty((w.decode.batch, w.Hq), dtype=torch.float32, device=dev)
    out, _ = mp.attn_decode(t["q"], t["k_pool"], t["v_pool"], t["block_tables"], t["block_starts"],
                            t["seq_lens"], t["q_pos"], rope, lse=lse)
    return out, lse


def test_noalloc_decode_matches_regular_on_calls_in_a_row(env):
    torch, mp, fn, dev = env
    cases = [W.long_decode(40, "bf16", B=2, n_spans=3, span_tokens=4096, pool_spans=4),    # 16 counters
             W.rag_decode(41, "bf16", B=5, n_spans=5, span_tokens=256, pool_spans=12, tail_tokens=99),
             W.rag_decode(42, "f32", B=12, n_spans=4, span_tokens=256, pool_spans=10, tail_tokens=37),
             W.rag_decode(43, "f32", B=3, n_spans=6, span_tokens=512, pool_spans=9, tail_tokens=5)]
    for w in cases:
        t = upload_decode(w, torch, dev)
        rope = mp.rope_table(w.max_pos, w.d, w.rope_base, device=dev)
        n_ws = mp.decode_workspace_size(w.decode.batch, w.Hq, w.Hkv, w.d, t["block_tables"].shape[1])
        assert n_ws > 0, "the case must use split-KV scratch"
        o1, l1 = _noalloc(env, w, t, rope)
        o2, l2 = _regular(env, w, t, rope)
        torch.cuda.synchronize()
        a, b = o1.float().cpu().numpy(), o2.float().cpu().numpy()
        assert np.all(np.isfinite(a))
        tol = TOL[w.dtype]
        diff = np.abs(a - b)
        assert diff.max() <= tol["max_abs"] and diff.mean() <= tol["mean_abs"]
        assert np.abs(l1.cpu().numpy() - l2.cpu().numpy()).max() <= tol["lse"]
        assert mp.device_error() == 0
    # the third call's counters (96 of them: 512 bytes) covered bytes that the
    # second call (40 counters: 256 bytes) had filled with partial results
    assert -(-12 * 8 * 4 // 256) * 256 > -(-5 * 8 * 4 // 256) * 256


def test_noalloc_rejects_shapes_beyond_the_fixed_scratch(env):
    torch, mp, fn, dev = env
    limit = 16 << 20
    # find a (batch, q heads, kv heads, table width) whose split-KV partials
    # exceed the fixed scratch on this device; the call must refuse it before
    # touching the device (all pointers below are never dereferenced)
    cands = [(b, hq, hkv, mb) for b in (8, 16, 32, 48, 64, 96, 128)
             for hq, hkv in ((64, 8), (128, 8), (32, 2), (16, 1))
             for mb in (1 << 12, 3 << 12, 1 << 14, 3 << 14, 1 << 16, 5 << 14)]
    big = max(cands, key=lambda c: mp.decode_workspace_size(c[0], c[1], c[2], 128, c[3]))
    assert mp.decode_workspace_size(big[0], big[1], big[2], 128, big[3]) > limit
    b, hq, hkv, mb = big
    kv = mp._KV(0x1000, 0x2000, 16, hkv, 16, 128)
    rp = mp._Rope(0x3000, 1 << 20, 128, None, 0xA000)
    db = mp._Decode(0x4000, 0x5000, 0x6000, 0x7000, 0x8000, b, mb, 0x9000, None)
    assert fn(mp.BF16, hq, ctypes.byref(kv), ctypes.byref(rp), ctypes.byref(db), 0.0, None) == 3
