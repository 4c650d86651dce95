"""The library's block-hash chain and prefix cache (host C++, through the C ABI)
against the oracle: bit-exact hashes and identical block tables.  CPU only."""

import numpy as np
import pytest

import oracle
import oracle.blockhash as bh
import position_independent_kv_paged_gb300 as mp
import workloads as W
from position_independent_kv_paged_gb300 import _build

SSEP, PDEP = 128001, 128002


@pytest.fixture(scope="module", autouse=True)
def lib():
    _build.build()
    return mp.load()


def _random_prompt(rng, n_spans, spans, bs, tail):
    """System block, then spans (each SSEP-led, padded to the block size), then
    a PDEP-led question and a ragged tail."""
    toks = list(rng.integers(0, 1000, size=bs))
    for s in rng.choice(len(spans), size=n_spans, replace=False):
        toks += spans[s]
    q = [PDEP] + list(rng.integers(0, 1000, size=bs - 1))
    return toks + q + list(rng.integers(0, 1000, size=tail))


def _spans(rng, n, bs):
    out = []
    for _ in range(n):
        nb = int(rng.integers(1, 4))
        body = [SSEP] + list(rng.integers(0, 1000, size=nb * bs - 1))
        out.append(body)
    return out


@pytest.mark.parametrize("bs", [4, 16])
def test_hashes_bit_exact(bs):
    rng = np.random.default_rng(bs)
    spans = _spans(rng, 6, bs)
    for k in range(20):
        toks = _random_prompt(rng, int(rng.integers(0, 5)), spans, bs, int(rng.integers(0, bs)))
        h0 = int(rng.integers(0, 1 << 62))
        got = mp.block_hashes(toks, bs, SSEP, PDEP, h0)
        want = bh.block_hashes(toks, bs, SSEP, PDEP, h0)
        assert [int(x) for x in got] == want


def test_hash_validation():
    with pytest.raises(mp.MiniPICError):
        mp.block_hashes([1, 2, 3], 0, SSEP, PDEP)
    assert mp.block_hashes([], 4, SSEP, PDEP).size == 0
    assert mp.block_hashes([1, 2, 3], 4, SSEP, PDEP).size == 0


def test_prefix_cache_matches_the_oracle_through_churn():
    """Random requests arrive, are assigned, and leave; both caches go through
    the same calls and must hand out the same blocks, starts and miss flags,
    and fail (pool full) on the same requests."""
    rng = np.random.default_rng(1)
    bs = 16
    spans = _spans(rng, 10, bs)
    ref, lib_c = bh.PrefixCache(24), mp.PrefixCache(24)
    live = []
    fails = hits = 0
    for step in range(400):
        if live and (len(live) > 6 or rng.random() < 0.4):
            tab = live.pop(int(rng.integers(0, len(live))))
            ref.release(tab)
            lib_c.release(tab)
            continue
        toks = _random_prompt(rng, int(rng.integers(0, 4)), spans, bs, int(rng.integers(0, bs)))
        hashes = bh.block_hashes(toks, bs, SSEP, PDEP, 7)
        n_blocks = -(-len(toks) // bs)
        r = ref.assign(hashes, n_blocks, bs)
        if r is None:
            with pytest.raises(mp.MiniPICError) as e:
                lib_c.assign(np.array(hashes, dtype=np.uint64), n_blocks, bs)
            assert e.value.status == 6
            fails += 1
            continue
        t, s, n = lib_c.assign(np.array(hashes, dtype=np.uint64), n_blocks, bs)
        assert np.array_equal(t, r[0]) and np.array_equal(s, r[1]) and np.array_equal(n, r[2])
        hits += int((n == 0).sum())
        live.append(t)
    assert fails > 0 and hits > 0  # both the full pool (with its roll-back) and cache hits were exercised
    lib_c.close()


def test_release_rejects_bad_ids_without_change():
    c = mp.PrefixCache(4)
    t, _, _ = c.assign(np.array([5, 6], dtype=np.uint64), 2, 16)
    with pytest.raises(mp.MiniPICError):
        c.release([t[0], t[0]])          # one reference only
    with pytest.raises(mp.MiniPICError):
        c.release([9])
    c.release([t[0]])
    _, _, n = c.assign(np.array([5], dtype=np.uint64), 1, 16)
    assert n[0] == 0                      # still cached after the failed releases


def test_shared_span_blocks_attend_like_private_copies():
    """Two prompts share an SSEP span at different offsets: the cache gives
    them the same physical blocks at different starts, and attention over those
    tables (oracle) equals attention over private copies of the span's keys."""
    rng = np.random.default_rng(3)
    bs = 16
    span = [SSEP] + list(rng.integers(0, 1000, size=2 * bs - 1))
    p1 = list(rng.integers(0, 1000, size=bs)) + span + [PDEP] + list(rng.integers(0, 1000, size=20))
    p2 = list(rng.integers(0, 1000, size=3 * bs)) + span + [PDEP] + list(rng.integers(0, 1000, size=9))
    c = mp.PrefixCache(32)
    tabs, starts = [], []
    for p in (p1, p2):
        t, s, _ = c.assign(mp.block_hashes(p, bs, SSEP, PDEP), -(-len(p) // bs), bs)
        tabs.append(t)
        starts.append(s)
    assert list(tabs[0][1:3]) == list(tabs[1][3:5]) and starts[0][1] != starts[1][3]
    # keys and values per physical block (the pool the tables index)
    Hq, Hkv, d = 4, 2, 64
    nblk = int(max(t.max() for t in tabs)) + 1
    k = rng.standard_normal((nblk, Hkv, bs, d)).astype(np.float32)
    v = rng.standard_normal((nblk, Hkv, bs, d)).astype(np.float32)
    mb = max(len(t) for t in tabs)
    bt = np.full((2, mb), -1, dtype=np.int32)
    st = np.zeros((2, mb), dtype=np.int32)
    for r in range(2):
        bt[r, :len(tabs[r])], st[r, :len(starts[r])] = tabs[r], starts[r]
    seq = np.array([len(p1), len(p2)], dtype=np.int32)
    q = rng.standard_normal((2, Hq, d)).astype(np.float32)
    w = W.Workload("shared", "f32", Hq, Hkv, d, bs, 10000.0, 200, W.PagedKV(k, v),
                   decode=W.DecodeBatch(q, bt, st, seq, seq.copy()))
    out, _ = oracle.decode(w)
    # private copies: every request gets its own blocks
    kp = np.concatenate([k[bt[r, :len(tabs[r])]] for r in range(2)])
    vp = np.concatenate([v[bt[r, :len(tabs[r])]] for r in range(2)])
    bt2 = np.full((2, mb), -1, dtype=np.int32)
    bt2[0, :len(tabs[0])] = np.arange(len(tabs[0]))
    bt2[1, :len(tabs[1])] = len(tabs[0]) + np.arange(len(tabs[1]))
    w2 = W.Workload("private", "f32", Hq, Hkv, d, bs, 10000.0, 200, W.PagedKV(kp, vp),
                    decode=W.DecodeBatch(q, bt2, st, seq, seq.copy()))
    out2, _ = oracle.decode(w2)
    assert np.abs(out - out2).max() < 1e-12
