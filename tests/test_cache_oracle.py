"""Pins of the cache-append oracle (oracle.cache) against what the MiniPIC
summary fixes (section 2.1: the cache holds unrotated keys) and against the
attention gather: appended rows read back unchanged, other slots untouched,
stored bytes independent of the position, and rebuilding the workloads' own
chunks reproduces their pools.  Planted mistakes must fail these checks."""

import numpy as np
import pytest

import oracle
from oracle import cache
import workloads as W


def _append_case(seed=0, dtype="bf16"):
    return W.append_case(seed, dtype)


def _slots_written(w, cu, kv_start):
    d = w.decode
    out = set()
    for r in range(len(cu) - 1):
        for i in range(int(cu[r + 1] - cu[r])):
            j = int(kv_start[r]) + i
            out.add((int(d.block_tables[r][j // 16]), j % 16))
    return out


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_appended_rows_read_back_and_nothing_else_moves(dtype):
    w, k_new, v_new, cu, kv_start = _append_case(1, dtype)
    d = w.decode
    k2, v2 = cache.append(w.kv.k_pool, w.kv.v_pool, k_new, v_new, cu, kv_start, d.block_tables)
    for r in range(len(cu) - 1):
        n = int(cu[r + 1] - cu[r])
        np.testing.assert_array_equal(cache.gather(k2, d.block_tables[r], int(kv_start[r]), n), k_new[cu[r]:cu[r + 1]])
        np.testing.assert_array_equal(cache.gather(v2, d.block_tables[r], int(kv_start[r]), n), v_new[cu[r]:cu[r + 1]])
    written = _slots_written(w, cu, kv_start)
    for b in range(k2.shape[0]):
        for s in range(16):
            if (b, s) not in written:
                assert np.array_equal(k2[b, :, s], w.kv.k_pool[b, :, s])
                assert np.array_equal(v2[b, :, s], w.kv.v_pool[b, :, s])
    # the old keys of every request still read back as before
    for r in range(len(cu) - 1):
        n_old = int(kv_start[r])
        np.testing.assert_array_equal(cache.gather(k2, d.block_tables[r], 0, n_old),
                                      cache.gather(w.kv.k_pool, d.block_tables[r], 0, n_old))


def test_rebuilding_own_chunks_reproduces_the_pools():
    """The prefill workloads' chunk keys, cleared and appended back at
    kv_len - q_len, give the generator's pools byte for byte."""
    w = W.rag_prefill(2, B=3, n_spans=2, span_tokens=64, pool_spans=4, q_len=40)
    p = w.prefill
    q_lens = np.diff(p.cu_q_lens).astype(np.int64)
    kv_start = p.kv_lens.astype(np.int64) - q_lens
    cu = np.concatenate([[0], np.cumsum(q_lens)])
    k_new = np.concatenate([cache.gather(w.kv.k_pool, p.block_tables[r], int(kv_start[r]), int(q_lens[r]))
                            for r in range(p.batch)])
    v_new = np.concatenate([cache.gather(w.kv.v_pool, p.block_tables[r], int(kv_start[r]), int(q_lens[r]))
                            for r in range(p.batch)])
    kc, vc = w.kv.k_pool.copy(), w.kv.v_pool.copy()
    for r in range(p.batch):
        for j in range(int(kv_start[r]), int(p.kv_lens[r])):
            kc[p.block_tables[r][j // 16], :, j % 16] = 0
            vc[p.block_tables[r][j // 16], :, j % 16] = 0
    assert not np.array_equal(kc, w.kv.k_pool)
    k2, v2 = cache.append(kc, vc, k_new, v_new, cu, kv_start, p.block_tables)
    assert np.array_equal(k2, w.kv.k_pool) and np.array_equal(v2, w.kv.v_pool)
    # and the attention over the rebuilt cache is the attention over the original
    w2 = W.Workload(**{**w.__dict__, "kv": W.PagedKV(**{**w.kv.__dict__, "k_pool": k2, "v_pool": v2})})
    a, _ = oracle.prefill(w, requests=[1])
    b, _ = oracle.prefill(w2, requests=[1])
    assert np.array_equal(a, b, equal_nan=True) and np.isfinite(a).any()


def test_stored_keys_do_not_depend_on_the_position():
    """The same key appended at two key indices with different block starts
    is stored as the same bits (no rotation on the way into the cache)."""
    w, k_new, v_new, cu, kv_start = _append_case(3, "f32")
    d = w.decode
    k_same = k_new.copy()
    k_same[cu[2]] = k_same[cu[0]]  # request 2's first new key := request 0's first
    assert d.block_starts[0][int(kv_start[0]) // 16] != d.block_starts[2][int(kv_start[2]) // 16] or \
        int(kv_start[0]) % 16 != int(kv_start[2]) % 16
    k2, _ = cache.append(w.kv.k_pool, w.kv.v_pool, k_same, v_new, cu, kv_start, d.block_tables)
    a = cache.gather(k2, d.block_tables[0], int(kv_start[0]), 1)[0]
    b = cache.gather(k2, d.block_tables[2], int(kv_start[2]), 1)[0]
    assert np.array_equal(a, b) and np.array_equal(a, k_new[cu[0]])


def test_empty_append_changes_nothing():
    w, k_new, v_new, cu, kv_start = _append_case(4, "bf16")
    cu0 = np.zeros(len(cu), dtype=np.int64)
    k2, v2 = cache.append(w.kv.k_pool, w.kv.v_pool, k_new[:0], v_new[:0], cu0, kv_start, w.decode.block_tables)
    assert np.array_equal(k2, w.kv.k_pool) and np.array_equal(v2, w.kv.v_pool)


# ---------------------------------------------------------------- planted mistakes

def _append_wrong_block(k_pool, v_pool, k_new, v_new, cu, kv_start, tables):
    k = k_pool.copy()
    v = v_pool.copy()
    for r in range(len(cu) - 1):
        for i in range(int(cu[r + 1] - cu[r])):
            j = int(kv_start[r]) + i
            k[tables[r][(j // 8) % len(tables[r])], :, j % 16] = k_new[cu[r] + i]  # block index off by a factor 2
            v[tables[r][(j // 8) % len(tables[r])], :, j % 16] = v_new[cu[r] + i]
    return k, v


def _append_rotated(w, k_new, cu, kv_start):
    """A cache that stores R_pi k (the pre-rotated design the method replaces)."""
    d = w.decode
    k = w.kv.k_pool.copy()
    for r in range(len(cu) - 1):
        for i in range(int(cu[r + 1] - cu[r])):
            j = int(kv_start[r]) + i
            pos = int(d.block_starts[r][j // 16]) + j % 16
            k[d.block_tables[r][j // 16], :, j % 16] = oracle.rope_rotate(k_new[cu[r] + i], np.full(1, pos), w.rope_base)
    return k


def test_planted_mistakes_are_caught():
    w, k_new, v_new, cu, kv_start = _append_case(5, "f32")
    d = w.decode
    kw, _ = _append_wrong_block(w.kv.k_pool, w.kv.v_pool, k_new, v_new, cu, kv_start, d.block_tables)
    r = 0
    n = int(cu[r + 1] - cu[r])
    assert not np.array_equal(cache.gather(kw, d.block_tables[r], int(kv_start[r]), n), k_new[cu[r]:cu[r + 1]])
    kr = _append_rotated(w, k_new, cu, kv_start)
    got = cache.gather(kr, d.block_tables[2], int(kv_start[2]), 3)
    assert not np.allclose(got, k_new[cu[2]:cu[2] + 3])


# ---------------------------------------------------------------- host offload

def _offload_case(dtype="bf16"):
    """rag-like decode over shared spans; the blocks of request 0 go to the host
    and come back to fresh physical ids."""
    w = W.rag_decode(6, dtype, B=4, Hq=8, Hkv=2, d=64, system_tokens=32, n_spans=3, span_tokens=64,
                     pool_spans=6, tail_tokens=32)
    d = w.decode
    n0 = -(-int(d.seq_lens[0]) // 16)
    old = np.unique(d.block_tables[0, :n0])
    nb = w.kv.num_blocks
    new = np.arange(nb, nb + len(old))  # fresh ids past the current pool
    grow = lambda a: np.concatenate([a, np.zeros((len(old),) + a.shape[1:], dtype=a.dtype)])
    return w, old, new, grow(w.kv.k_pool), grow(w.kv.v_pool)


def test_swap_round_trip_is_identity():
    w, old, new, kp, vp = _offload_case()
    kh, vh = cache.swap_out(kp, vp, old)
    kc, vc = kp.copy(), vp.copy()
    kc[old] = 0
    vc[old] = 0
    k2, v2 = cache.swap_in(kc, vc, kh, vh, old)
    assert np.array_equal(k2, kp) and np.array_equal(v2, vp)


def test_relocated_blocks_need_no_position_fixup():
    """Blocks swapped out and back in at other physical ids, with the tables
    remapped and block_starts untouched, give the same attention bit for bit."""
    w, old, new, kp, vp = _offload_case()
    ref, ref_lse = oracle.decode(w)
    kh, vh = cache.swap_out(kp, vp, old)
    kc, vc = kp.copy(), vp.copy()
    kc[old] = 0  # the old copies are gone
    vc[old] = 0
    k2, v2 = cache.swap_in(kc, vc, kh, vh, new)
    d = w.decode
    d2 = W.DecodeBatch(q=d.q, block_tables=cache.remap_tables(d.block_tables, old, new).astype(np.int32),
                       block_starts=d.block_starts, seq_lens=d.seq_lens, q_pos=d.q_pos)
    w2 = W.Workload(**{**w.__dict__, "kv": W.PagedKV(k2, v2), "decode": d2})
    out, lse = oracle.decode(w2)
    assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)
    # planted mistake: the blocks come back in the wrong order
    k3, v3 = cache.swap_in(kc, vc, kh, vh, new[::-1].copy())
    w3 = W.Workload(**{**w.__dict__, "kv": W.PagedKV(k3, v3), "decode": d2})
    bad, _ = oracle.decode(w3, requests=[0])
    assert not np.allclose(bad[0], ref[0])
