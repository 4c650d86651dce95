"""CPU checks of the coded inputs that the exact-indexing GPU tests use: the
oracle's outputs on them spell out the oracle's own key index map as integer
counts, and a planted indexing mistake in the oracle changes those counts."""

import numpy as np
import pytest

import oracle
import oracle.attention as oatt
from index_codes import (ALIGNED, aligned_decode, counts, counts_from_indices, phase_margin, zero_query_decode,
                         zero_query_prefill)


def _decode_counts(w, out):
    dec = w.decode
    got, exp = [], []
    for r in range(dec.batch):
        n = int(dec.seq_lens[r])
        if n == 0:
            continue
        phys, slot, _ = oracle.key_index_map(dec.block_tables[r], dec.block_starts[r], n, 16)
        for h in range(w.Hq):
            c, frac = counts(out[r, h], n)
            got.append((c, frac))
            exp.append(counts_from_indices(phys, slot, w.d))
    return got, exp


@pytest.mark.parametrize("dtype,Hq,Hkv,d", [("f32", 8, 2, 128), ("bf16", 6, 2, 64)])
def test_zero_query_decode_counts_equal_the_index_map(dtype, Hq, Hkv, d):
    w = zero_query_decode(3, dtype, Hq, Hkv, d, [0, 1, 15, 17, 300])
    out, lse = oracle.decode(w)
    got, exp = _decode_counts(w, out)
    for (c, frac), e in zip(got, exp):
        assert frac < 1e-9 and np.array_equal(c, e)
    G = Hq // Hkv
    for r in range(1, w.decode.batch):
        for h in range(Hq):
            assert abs(out[r, h, -1] - (h // G + 1)) < 1e-12


def test_zero_query_prefill_counts_equal_the_index_map():
    w = zero_query_prefill(4, 8, 2, 128, kv_lens=[1, 40, 300], q_lens=[1, 40, 37])
    out, _ = oracle.prefill(w)
    p = w.prefill
    for r in range(p.batch):
        q0, q1 = int(p.cu_q_lens[r]), int(p.cu_q_lens[r + 1])
        kv = int(p.kv_lens[r])
        phys, slot, _ = oracle.key_index_map(p.block_tables[r], p.block_starts[r], kv, 16)
        for i in range(q1 - q0):
            n = kv - (q1 - q0) + i + 1
            c, frac = counts(out[q0 + i, 0], n)
            assert frac < 1e-9 and np.array_equal(c, counts_from_indices(phys[:n], slot[:n], w.d))


def test_aligned_decode_scores_every_key_alike():
    c = ALIGNED
    M = c["M"]
    assert M * (1.0 - phase_margin(c["d"], 10000.0, c["n_pairs"], 2 * c["max_pos"])) >= 25.0
    w = aligned_decode()
    out, lse = oracle.decode(w)
    got, exp = _decode_counts(w, out)
    for (cnt, frac), e in zip(got, exp):
        assert frac < 1e-4 and np.array_equal(cnt, e)
    n = np.asarray(c["seq"], dtype=np.float64)[:, None]
    assert np.abs(lse - (M + np.log(n))).max() < 1e-6 * M


def test_phase_margin_closed_forms():
    # one frequency, theta_0 = 1: the largest cos(delta) over delta = 1..6 is cos(6) (6 is nearest 2 pi)
    assert phase_margin(64, 10000.0, 1, 6) == pytest.approx(np.cos(6.0), abs=1e-15)
    assert phase_margin(64, 10000.0, 1, 1) == pytest.approx(np.cos(1.0), abs=1e-15)


def _shifted_positions(table_row, start_row, n_keys, bs):
    phys, slot, pos = oracle.key_index_map(table_row, start_row, n_keys, bs)
    pos = pos.copy()
    pos[n_keys // 2:] += 1  # keys in the second half rotated one position late
    return phys, slot, pos


def _wrong_slot(table_row, start_row, n_keys, bs):
    phys, slot, pos = oracle.key_index_map(table_row, start_row, n_keys, bs)
    return phys, (slot + 1) % bs, pos


def _wrong_block(table_row, start_row, n_keys, bs):
    phys, slot, pos = oracle.key_index_map(table_row, start_row, n_keys, bs)
    return (phys + 1) % 64, slot, pos


def test_aligned_decode_catches_a_planted_position_mistake(monkeypatch):
    w = aligned_decode()  # aligned for the true positions
    monkeypatch.setattr(oatt, "key_index_map", _shifted_positions)
    out, _ = oracle.decode(w)
    monkeypatch.undo()
    got, exp = _decode_counts(w, out)
    assert any(not np.array_equal(cnt, e) for (cnt, _), e in zip(got, exp))


def test_aligned_decode_catches_a_planted_query_position_mistake():
    w = aligned_decode()
    w.decode.q_pos = w.decode.q_pos + 1
    _, lse = oracle.decode(w)
    n = np.asarray(ALIGNED["seq"], dtype=np.float64)[:, None]
    assert np.abs(lse - (ALIGNED["M"] + np.log(n))).min() > 1.0


@pytest.mark.parametrize("mutant", [_wrong_slot, _wrong_block])
def test_zero_query_decode_catches_a_planted_gather_mistake(monkeypatch, mutant):
    w = zero_query_decode(3, "f32", 8, 2, 128, [0, 1, 15, 17, 300])
    monkeypatch.setattr(oatt, "key_index_map", mutant)
    out, _ = oracle.decode(w)
    monkeypatch.undo()
    got, exp = _decode_counts(w, out)
    assert any(not np.array_equal(cnt, e) for (cnt, _), e in zip(got, exp))
