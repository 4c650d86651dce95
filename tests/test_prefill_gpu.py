"""Chunked-prefill parity: the tcgen05 CUDA path (through the C ABI) against the
CPU oracle, on RAG-shaped, causal-from-zero and irregular inputs."""

import os

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import TOL, compare, compare_lse, upload_prefill
from oracle_pool import OraclePool

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
    return torch, mp, torch.device("cuda:0")


def run_prefill(env, w):
    torch, mp, dev = env
    p = w.prefill
    t = upload_prefill(w, torch, dev)
    rope = mp.rope_table(w.max_pos, w.d, w.rope_base, device=dev)
    lse = torch.full((int(p.cu_q_lens[-1]), w.Hq), float("nan"), dtype=torch.float32, device=dev)
    max_q = int(np.diff(p.cu_q_lens).max()) if p.batch else 1
    out, _ = mp.attn_prefill(t["q"], t["cu_q_lens"], t["q_pos"], t["k_pool"], t["v_pool"], t["block_tables"],
                             t["block_starts"], t["kv_lens"], rope, max_q_len=max_q, lse=lse)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def test_rag_prefill_scaled(env):
    w = W.rag_prefill(1, B=3, n_spans=2, span_tokens=256, pool_spans=6, q_len=200)
    out, lse = run_prefill(env, w)
    ref, rl = oracle.prefill(w)
    compare(out, ref, "bf16", "rag_prefill small")
    compare_lse(lse, rl, "bf16", "rag_prefill small")
    assert env[1].device_error() == 0


@pytest.mark.parametrize("Hq,Hkv", [(28, 4), (8, 8), (16, 1), (32, 8)])
def test_causal_span_prefill_from_zero(env, Hq, Hkv):
    w = W.mixed_batch(2, n_prefill=3, chunk=300, n_decode=0, Hq=Hq, Hkv=Hkv)
    out, lse = run_prefill(env, w)
    ref, rl = oracle.prefill(w)
    compare(out, ref, "bf16", f"span prefill {Hq}/{Hkv}")
    compare_lse(lse, rl, "bf16", "span prefill")


@pytest.mark.parametrize("Hq,Hkv,d", [(8, 2, 128), (12, 4, 64), (7, 1, 128), (4, 4, 64)])
def test_irregular_prefill(env, Hq, Hkv, d):
    w = W.irregular_prefill(5 + Hq, "bf16", kv_lens=[1, 17, 300, 129, 513], q_lens=[1, 5, 300, 1, 77], Hq=Hq,
                            Hkv=Hkv, d=d, max_pos=60000)
    out, lse = run_prefill(env, w)
    ref, rl = oracle.prefill(w)
    compare(out, ref, "bf16", f"irregular prefill {Hq}/{Hkv}/{d}")
    compare_lse(lse, rl, "bf16", "irregular prefill")


def test_prefill_rejects_f32(env):
    torch, mp, dev = env
    w = W.irregular_prefill(3, "f32", kv_lens=[20], q_lens=[4], Hq=4, Hkv=2, d=128, max_pos=100)
    with pytest.raises(mp.MiniPICError) as e:
        run_prefill(env, w)
    assert e.value.status == 2


def test_prefill_flags_bad_block_ids(env):
    torch, mp, dev = env
    w = W.irregular_prefill(8, "bf16", kv_lens=[100, 60], q_lens=[30, 60], Hq=4, Hkv=2, d=128, max_pos=1000)
    mp.device_error(clear=True)
    w.prefill.block_tables[1, 2] = 10 ** 6
    out, _ = run_prefill(env, w)
    assert mp.device_error(clear=True) & 1
    assert np.all(np.isfinite(out))


@pytest.mark.parametrize("idx,sample", [(2, list(range(8))), (4, [0, 3, 7, 12, 15])])
def test_full_size_prefill(env, idx, sample):
    """The full RAG prefill (all 8 requests) and 5 of the mixed batch's 16 span
    prefills, against the oracle run on every host core."""
    w = W.config(idx)
    if idx == 4:
        w.decode = None
    out, lse = run_prefill(env, w)
    with OraclePool(w, n_workers=min(len(sample), os.cpu_count() or 1)) as op:
        ref, rl = op.prefill(sample)
    rows = np.concatenate([np.arange(w.prefill.cu_q_lens[r], w.prefill.cu_q_lens[r + 1]) for r in sample])
    compare(out[rows], ref[rows], "bf16", f"config {idx} sampled")
    compare_lse(lse[rows], rl[rows], "bf16", f"config {idx} sampled")
    assert np.all(np.isfinite(out))
    assert env[1].device_error() == 0


def test_prerotated_prefill_equals_oracle_on_private_copies(env):
    """The rotation-free prefill over a cache pre-rotated on the host (every
    block used by one request) equals the oracle over the unrotated cache."""
    torch, mp, dev = env
    # private blocks only (each pre-rotated once); rows attend 401..600 keys
    w = W.build_workload("private_prefill", 9, "bf16", Hq=8, Hkv=2, d=128, rope_base=500000.0, pool_spans=0,
                         span_tokens=16, prefill_requests=[([("own", 600)], 200)] * 3)
    ref, rl = oracle.prefill(w)
    p = w.prefill
    k = oracle.widen(w.kv.k_pool, "bf16").copy()
    q = oracle.widen(p.q, "bf16").copy()
    for r in range(p.batch):
        phys, slot, pos = oracle.key_index_map(p.block_tables[r], p.block_starts[r], int(p.kv_lens[r]), 16)
        for g in range(w.Hkv):
            k[phys, g, slot] = oracle.rope_rotate(k[phys, g, slot], pos, w.rope_base)
        q0, q1 = int(p.cu_q_lens[r]), int(p.cu_q_lens[r + 1])
        for h in range(w.Hq):
            q[q0:q1, h] = oracle.rope_rotate(q[q0:q1, h], p.q_pos[q0:q1], w.rope_base)
    w.kv.k_pool = W.to_bf16_bits(k.astype(np.float32))
    p.q = W.to_bf16_bits(q.astype(np.float32))
    t = upload_prefill(w, torch, dev)
    out, _ = mp.attn_prefill_prerotated(t["q"], t["cu_q_lens"], t["q_pos"], t["k_pool"], t["v_pool"],
                                        t["block_tables"], t["block_starts"], t["kv_lens"], max_q_len=200)
    torch.cuda.synchronize()
    compare(out.float().cpu().numpy(), ref, "bf16", "prerotated prefill")


@pytest.mark.parametrize("Hq,Hkv,d", [(32, 8, 128), (12, 4, 64)])
def test_prefill_with_empty_chunks(env, Hq, Hkv, d):
    """Requests without query tokens sit between others: their query-tile pairs
    do nothing and the other requests' rows are unaffected."""
    w = W.irregular_prefill(40 + d, "bf16", kv_lens=[16, 40, 700, 5, 64, 9], q_lens=[0, 1, 333, 0, 64, 9], Hq=Hq,
                            Hkv=Hkv, d=d, max_pos=30000)
    out, lse = run_prefill(env, w)
    ref, rl = oracle.prefill(w)
    compare(out, ref, "bf16", f"prefill with empty chunks {Hq}/{Hkv}/{d}")
    compare_lse(lse, rl, "bf16", "prefill with empty chunks")
    assert env[1].device_error() == 0


@pytest.mark.parametrize("case", ["rag", "short_items"])
def test_prefill_repeats_bit_for_bit(env, case):
    """Every launch computes the same sums in the same order, so repeated calls
    agree bit for bit; a race between the two CTAs of a pair (an operand read
    before its writer finished) shows up here as a difference between calls."""
    if case == "rag":
        w = W.rag_prefill(3, B=4, n_spans=3, span_tokens=512, pool_spans=8, q_len=300)
    else:  # many query-tile pairs with one or two key tiles each
        w = W.mixed_batch(7, n_prefill=6, chunk=300, n_decode=0, Hq=28, Hkv=4)
    first, first_lse = run_prefill(env, w)
    for _ in range(4):
        out, lse = run_prefill(env, w)
        assert np.array_equal(out, first) and np.array_equal(lse, first_lse, equal_nan=True)
    assert env[1].device_error() == 0


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("where", ["key", "query"])
def test_fp16_range_overflow_is_flagged(env, d, where):
    """The QK^T operands are fp16: a rotated key element, or a rotated and
    scaled query element, beyond +-65504 sets MINIPIC_DEVERR_RANGE (16).  Rows
    that read the element are undefined; every other row stays finite and
    matches the oracle."""
    torch, mp, dev = env
    w = W.irregular_prefill(77 + d, "bf16", kv_lens=[300, 200, 90], q_lens=[200, 200, 90], Hq=8, Hkv=2, d=d,
                            max_pos=30000)
    p = w.prefill
    G = w.Hq // w.Hkv
    big = W.to_bf16_bits(np.array([2.0e6], dtype=np.float32))[0]  # > 65504 / (scale log2 e) as well
    bad = np.zeros((int(p.cu_q_lens[-1]), w.Hq), dtype=bool)  # (query row, head) that read the element
    if where == "key":
        j0 = 250  # key 250 of request 0: block 15, slot 10, kv head 1, element 3
        phys, slot = int(p.block_tables[0, j0 // 16]), j0 % 16
        w.kv.k_pool[phys, 1, slot, 3] = big
        for r in range(p.batch):
            kv, q0, q1 = int(p.kv_lens[r]), int(p.cu_q_lens[r]), int(p.cu_q_lens[r + 1])
            ph, sl, _ = oracle.key_index_map(p.block_tables[r], p.block_starts[r], kv, 16)
            hits = np.nonzero((ph == phys) & (sl == slot))[0]
            for i in range(q1 - q0):
                if hits.size and hits.min() <= kv - (q1 - q0) + i:
                    bad[q0 + i, G:2 * G] = True
    else:
        row = int(p.cu_q_lens[1]) + 7  # request 1, chunk query 7, head 5
        p.q[row, 5, 2] = big
        bad[row, 5] = True
    mp.device_error(clear=True)
    out, _ = run_prefill(env, w)
    assert mp.device_error(clear=True) & 16
    ref, _ = oracle.prefill(w)
    ok = ~bad
    assert ok.sum() > 0.5 * ok.size
    assert np.all(np.isfinite(out[ok]))
    compare(out[ok], ref[ok], "bf16", f"rows away from the {where} overflow")
    # the same inputs without the large element raise no flag
    w2 = W.irregular_prefill(77 + d, "bf16", kv_lens=[300, 200, 90], q_lens=[200, 200, 90], Hq=8, Hkv=2, d=d,
                             max_pos=30000)
    run_prefill(env, w2)
    assert mp.device_error(clear=True) == 0
