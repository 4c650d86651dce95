"""The seeded input generators hold the recipe the benchmark and the parity
tests rely on: shapes, sizes, sharing structure and positions of each
workload (no method arithmetic lives in ``workloads``)."""

import numpy as np
import pytest

import workloads as W

BS = 16


def _rows(bt, st, n_blocks):
    return [int(x) for x in bt[:n_blocks]], [int(x) for x in st[:n_blocks]]


def _assert_contiguous_positions(st, n_blocks):
    assert np.array_equal(st[:n_blocks], np.arange(n_blocks, dtype=np.int32) * BS)


@pytest.fixture(scope="module")
def rag_decode():
    return W.rag_decode(0)


def test_rag_decode_recipe(rag_decode):
    w = rag_decode
    d = w.decode
    assert (w.Hq, w.Hkv, w.d, w.block_size, w.rope_base, w.dtype) == (32, 8, 128, 16, 500000.0, "bf16")
    assert d.batch == 64 and np.all(d.seq_lens == 8192) and np.all(d.q_pos == 8192)
    assert w.kv.k_pool.dtype == np.uint16 and w.kv.k_pool.shape[1:] == (8, 16, 128)
    sys_ids = d.block_tables[0, :16]
    tails = set()
    span_hits = {}
    for r in range(d.batch):
        bt, st = d.block_tables[r], d.block_starts[r]
        assert bt.shape[0] >= 512 and np.all(bt[:512] >= 0)
        _assert_contiguous_positions(st, 512)
        # 256-token system prompt: the same physical blocks at offset 0 in every request
        assert np.array_equal(bt[:16], sys_ids)
        # 15 retrieved spans of 512 tokens (32 blocks), distinct within the request
        spans = [tuple(int(x) for x in bt[16 + 32 * k: 16 + 32 * (k + 1)]) for k in range(15)]
        assert len(set(spans)) == 15
        for sp in spans:
            span_hits[sp] = span_hits.get(sp, 0) + 1
        # 256 private tokens: blocks no other request reads
        tail = [int(x) for x in bt[496:512]]
        assert not tails.intersection(tail)
        tails.update(tail)
    # the span blocks and the private blocks are disjoint, spans never share blocks
    span_blocks = [b for sp in span_hits for b in sp]
    assert len(span_blocks) == len(set(span_blocks))
    assert not tails.intersection(span_blocks) and not tails.intersection(int(x) for x in sys_ids)
    # Zipf(1.1) over 256 spans: the most popular span is in most requests, and
    # shared spans sit at different offsets in different requests
    assert max(span_hits.values()) >= 32
    top = max(span_hits, key=span_hits.get)
    offsets = {int(np.nonzero(d.block_tables[r] == top[0])[0][0]) for r in range(d.batch)
               if top[0] in d.block_tables[r]}
    assert len(offsets) > 1
    assert w.unique_blocks == len(span_blocks) + len(tails) + 16


def test_rag_decode_no_sharing_control_reads_every_block_once():
    w = W.rag_decode(0, share=False, B=4)
    bt = w.decode.block_tables
    used = bt[bt >= 0]
    assert used.size == 4 * 512 and np.unique(used).size == used.size


def test_rag_prefill_recipe():
    w = W.rag_prefill(0)
    p = w.prefill
    assert (w.Hq, w.Hkv, w.d, w.rope_base) == (32, 8, 128, 500000.0)
    assert p.batch == 8 and np.all(np.diff(p.cu_q_lens) == 512) and np.all(p.kv_lens == 6656)
    own = set()
    for r in range(p.batch):
        bt, st = p.block_tables[r], p.block_starts[r]
        _assert_contiguous_positions(st, 416)
        spans = [tuple(int(x) for x in bt[64 * k: 64 * (k + 1)]) for k in range(6)]
        assert len(set(spans)) == 6
        chunk = [int(x) for x in bt[384:416]]
        assert not own.intersection(chunk)
        own.update(chunk)
        q = p.q_pos[p.cu_q_lens[r]:p.cu_q_lens[r + 1]]
        assert np.array_equal(q, np.arange(6144, 6656, dtype=np.int32))


def test_long_decode_recipe():
    w = W.long_decode(0)
    d = w.decode
    assert (w.Hq, w.Hkv, w.d, w.rope_base) == (64, 8, 128, 500000.0)
    assert d.batch == 8 and np.all(d.seq_lens == 131072)
    pool = set()
    for r in range(d.batch):
        _assert_contiguous_positions(d.block_starts[r], 8192)
        spans = [tuple(int(x) for x in d.block_tables[r, 256 * k: 256 * (k + 1)]) for k in range(32)]
        pool.update(spans)
    assert len(pool) <= 48


def test_mixed_batch_recipe():
    w = W.mixed_batch(0)
    p, d = w.prefill, w.decode
    assert (w.Hq, w.Hkv, w.d, w.rope_base) == (28, 4, 128, 1000000.0)
    assert p.batch == 16 and np.all(np.diff(p.cu_q_lens) == 2048) and np.all(p.kv_lens == 2048)
    for r in range(p.batch):
        assert np.array_equal(p.q_pos[p.cu_q_lens[r]:p.cu_q_lens[r + 1]], np.arange(2048, dtype=np.int32))
        _assert_contiguous_positions(p.block_starts[r], 128)
    assert d.batch == 128
    assert np.all(d.seq_lens >= 2048) and np.all(d.seq_lens <= 32768)
    for r in range(d.batch):
        L = int(d.seq_lens[r])
        nb = -(-L // BS)
        _assert_contiguous_positions(d.block_starts[r], nb)
        assert np.all(d.block_tables[r, :nb] >= 0)
        full = L // 1024
        spans = [tuple(int(x) for x in d.block_tables[r, 64 * k: 64 * (k + 1)]) for k in range(full)]
        assert len(set(spans)) == full


def test_tiny_decode_recipe():
    for dtype in ("f32", "bf16"):
        w = W.tiny_decode(0, dtype)
        d = w.decode
        assert (w.Hq, w.Hkv, w.d, w.rope_base) == (4, 2, 64, 10000.0)
        assert d.batch == 2 and np.all(d.seq_lens == 128) and w.kv.k_pool.shape[0] == 12
        pos = [{int(b): int(s) for b, s in zip(d.block_tables[r, :8], d.block_starts[r, :8])} for r in range(2)]
        shared = set(pos[0]) & set(pos[1])
        assert any(pos[0][b] != pos[1][b] for b in shared)


def test_generators_are_seeded():
    a, b, c = W.rag_prefill(3, B=2, q_len=64), W.rag_prefill(3, B=2, q_len=64), W.rag_prefill(4, B=2, q_len=64)
    for x, y in ((a.kv.k_pool, b.kv.k_pool), (a.kv.v_pool, b.kv.v_pool), (a.prefill.q, b.prefill.q),
                 (a.prefill.block_tables, b.prefill.block_tables)):
        assert np.array_equal(x, y)
    assert not np.array_equal(a.prefill.q, c.prefill.q)


def test_values_are_standard_normal_rounded_to_bf16():
    w = W.rag_prefill(0, B=2, n_spans=2, span_tokens=256, q_len=128)
    x = W.bf16_bits_to_f32(w.kv.k_pool).astype(np.float64).ravel()
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    # every stored value is exactly a bf16 number
    assert np.array_equal(W.to_bf16_bits(W.bf16_bits_to_f32(w.kv.k_pool)), w.kv.k_pool)
