"""Pins for the CPU oracle: it is checked against things other than itself.

* closed forms of the rotary table (p = 0, theta_0 = 1, theta_{d/4} = base^-1/2,
  unit norm, angle addition);
* hand-derived worked examples (tests/golden/worked_examples.json);
* brute force: explicit d x d rotation matrices, scalar loops, explicit softmax;
* equality with standard attention over private pre-rotated copies built with
  complex multiplication (the page's "algebraically equivalent to re-rotating
  the cache hit", MiniPIC summary section 2.1);
* the relative-position invariant and the all-zero-position reduction;
* block sharing at different offsets, with a negative control (a block
  pre-rotated once and reused at another offset must disagree, section 1);
* index pins (one key gives its value row exactly; q = 0 gives the mean);
* prefill rows equal decode with the matching key prefix;
* planted mistakes in the oracle are caught by at least one pin.
"""

import json
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle
import oracle.attention as oatt
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


# ---------------------------------------------------------------- helpers

def _w_from_case(c):
    pool_k = np.asarray(c["k_pool"], dtype=np.float32)
    pool_v = np.asarray(c["v_pool"], dtype=np.float32)
    kv = W.PagedKV(pool_k, pool_v)
    w = W.Workload(c["name"], "f32", c["Hq"], c["Hkv"], c["d"], c["block_size"],
                   c["rope_base"], 1 << 20, kv)
    bt = np.asarray(c["block_tables"], np.int32)
    st = np.asarray(c["block_starts"], np.int32)
    if c["kind"] == "decode":
        w.decode = W.DecodeBatch(np.asarray(c["q"], np.float32), bt, st,
                                 np.asarray(c["seq_lens"], np.int32), np.asarray(c["q_pos"], np.int32))
    else:
        w.prefill = W.PrefillBatch(np.asarray(c["q"], np.float32), np.asarray(c["cu_q_lens"], np.int32),
                                   np.asarray(c["q_pos"], np.int32), np.asarray(c["kv_lens"], np.int32), bt, st)
    return w


def _rot_matrix(p, d, base, cache):
    """Explicit d x d rotary matrix for position p (half-rotation pairing)."""
    key = (p, d, base)
    if key not in cache:
        h = d // 2
        M = np.zeros((d, d))
        for i in range(h):
            th = base ** (-2.0 * i / d)
            c, s = math.cos(p * th), math.sin(p * th)
            M[i, i] = c
            M[i, i + h] = -s
            M[i + h, i] = s
            M[i + h, i + h] = c
        cache[key] = M
    return cache[key]


def _val(w, arr):
    return W.bf16_bits_to_f32(arr).astype(np.float64) if w.dtype == "bf16" else np.asarray(arr, np.float64)


def _brute_rows(w, q_rows, q_positions, table, starts, n_keys_per_row, g):
    """Scalar-loop attention for query rows sharing one key list."""
    cache = {}
    d = w.d
    outs, lses = [], []
    for q, tq, nk in zip(q_rows, q_positions, n_keys_per_row):
        qr = _rot_matrix(int(tq), d, w.rope_base, cache) @ q
        scores, vals = [], []
        for j in range(nk):
            b, slot = j // w.block_size, j % w.block_size
            phys = int(table[b])
            pos = int(starts[b]) + slot
            k = _val(w, w.kv.k_pool[phys, g, slot])
            kr = _rot_matrix(pos, d, w.rope_base, cache) @ k
            s = 0.0
            for a in range(d):
                s += qr[a] * kr[a]
            scores.append(s / math.sqrt(d))
            vals.append(_val(w, w.kv.v_pool[phys, g, slot]))
        if not scores:
            outs.append(np.zeros(d))
            lses.append(-math.inf)
            continue
        m = max(scores)
        e = [math.exp(s - m) for s in scores]
        z = sum(e)
        o = np.zeros(d)
        for ej, v in zip(e, vals):
            o += (ej / z) * v
        outs.append(o)
        lses.append(m + math.log(z))
    return np.array(outs), np.array(lses)


def brute_decode(w):
    dec = w.decode
    G = w.Hq // w.Hkv
    out = np.zeros((dec.batch, w.Hq, w.d))
    lse = np.zeros((dec.batch, w.Hq))
    for r in range(dec.batch):
        for h in range(w.Hq):
            o, l = _brute_rows(w, [_val(w, dec.q[r, h])], [dec.q_pos[r]], dec.block_tables[r],
                               dec.block_starts[r], [int(dec.seq_lens[r])], h // G)
            out[r, h], lse[r, h] = o[0], l[0]
    return out, lse


def brute_prefill(w):
    pre = w.prefill
    G = w.Hq // w.Hkv
    tq = int(pre.cu_q_lens[-1])
    out = np.zeros((tq, w.Hq, w.d))
    lse = np.zeros((tq, w.Hq))
    for r in range(pre.batch):
        q0, q1 = int(pre.cu_q_lens[r]), int(pre.cu_q_lens[r + 1])
        ql, kv = q1 - q0, int(pre.kv_lens[r])
        for h in range(w.Hq):
            rows = [_val(w, pre.q[i, h]) for i in range(q0, q1)]
            nks = [kv - ql + i + 1 for i in range(ql)]
            o, l = _brute_rows(w, rows, pre.q_pos[q0:q1], pre.block_tables[r], pre.block_starts[r], nks, h // G)
            out[q0:q1, h], lse[q0:q1, h] = o, l
    return out, lse


def _complex_rotate(x, pos, d, base):
    """Rotate rows by multiplying (x_lo + i x_hi) with exp(i p theta)."""
    h = d // 2
    z = x[:, :h].astype(np.clongdouble) + 1j * x[:, h:].astype(np.clongdouble)
    i = np.arange(h, dtype=np.longdouble)
    th = np.power(np.longdouble(base), -2 * i / np.longdouble(d))
    ang = np.asarray(pos, dtype=np.longdouble)[:, None] * th[None, :]
    zr = z * np.exp(1j * ang.astype(np.clongdouble))
    return np.concatenate([zr.real, zr.imag], axis=1).astype(np.float64)


def _private_prerotated_decode(w, r, shared_override=None):
    """Standard attention over a private, pre-rotated, contiguous cache.

    ``shared_override`` = (phys, rotated_at_position) replaces the rotation of
    that physical block by one made at another offset (negative control)."""
    dec = w.decode
    G = w.Hq // w.Hkv
    L = int(dec.seq_lens[r])
    out = np.zeros((w.Hq, w.d))
    lse = np.zeros(w.Hq)
    qpos = int(dec.q_pos[r])
    for g in range(w.Hkv):
        ks, vs, ps = [], [], []
        for b in range(-(-L // w.block_size)):
            phys = int(dec.block_tables[r, b])
            n = min(w.block_size, L - b * w.block_size)
            k = _val(w, w.kv.k_pool[phys, g, :n])
            pos = int(dec.block_starts[r, b]) + np.arange(n)
            if shared_override and shared_override[0] == phys:
                pos = shared_override[1] + np.arange(n)
            ks.append(_complex_rotate(k, pos, w.d, w.rope_base))
            vs.append(_val(w, w.kv.v_pool[phys, g, :n]))
        K = np.concatenate(ks)
        V = np.concatenate(vs)
        for h in range(g * G, (g + 1) * G):
            q = _complex_rotate(_val(w, dec.q[r, h])[None, :], [qpos], w.d, w.rope_base)[0]
            s = K @ q / math.sqrt(w.d)
            out[h] = softmax(s) @ V
            lse[h] = logsumexp(s)
    return out, lse


def _scaled_irregular(seed, dtype="f32", **kw):
    return W.irregular_decode(seed, dtype, **kw)


# ---------------------------------------------------------------- table pins

@pytest.mark.parametrize("d,base", [(64, 10000.0), (128, 500000.0), (128, 1000000.0)])
def test_table_closed_forms(d, base):
    maxp = 131073
    T = oracle.rope_table(maxp, d, base)
    h = d // 2
    # p = 0: cos = 1, sin = 0 exactly
    assert np.all(T[0, :h] == 1.0) and np.all(T[0, h:] == 0.0)
    # theta_0 = base^0 = 1: column 0 is cos(p), sin(p)
    ps = np.array([1, 2, 7, 4095, 8192, 65536, 131072])
    for p in ps:
        assert abs(T[p, 0] - math.cos(p)) < 1e-12 and abs(T[p, h] - math.sin(p)) < 1e-12
    # theta_{d/4} = base^(-1/2)
    th = base ** -0.5
    for p in ps:
        assert abs(T[p, d // 4] - math.cos(p * th)) < 1e-12
        assert abs(T[p, h + d // 4] - math.sin(p * th)) < 1e-12
    # unit norm
    assert np.max(np.abs(T[:, :h] ** 2 + T[:, h:] ** 2 - 1.0)) < 1e-15
    # angle addition: R_a R_b = R_{a+b}
    rng = np.random.default_rng(1)
    a = rng.integers(0, maxp // 2, 200)
    b = rng.integers(0, maxp // 2, 200)
    ca, sa, cb, sb = T[a, :h], T[a, h:], T[b, :h], T[b, h:]
    assert np.max(np.abs(ca * cb - sa * sb - T[a + b, :h])) < 1e-14
    assert np.max(np.abs(sa * cb + ca * sb - T[a + b, h:])) < 1e-14


def test_rotation_is_complex_multiply_and_identity_at_zero():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((50, 128))
    pos = rng.integers(0, 131073, 50)
    np.testing.assert_allclose(oracle.rope_rotate(x, pos, 500000.0),
                               _complex_rotate(x, pos, 128, 500000.0), rtol=0, atol=1e-12)
    assert np.array_equal(oracle.rope_rotate(x, np.zeros(50, int), 500000.0), x)
    # rotation preserves the norm of every pair
    y = oracle.rope_rotate(x, pos, 500000.0)
    np.testing.assert_allclose(x[:, :64] ** 2 + x[:, 64:] ** 2, y[:, :64] ** 2 + y[:, 64:] ** 2, atol=1e-12)


# ---------------------------------------------------------------- worked examples

@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_worked_examples(case):
    w = _w_from_case(case)
    if case["kind"] == "decode":
        out, lse = oracle.decode(w)
    else:
        out, lse = oracle.prefill(w)
    np.testing.assert_allclose(out, np.asarray(case["expect_out"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, np.asarray(case["expect_lse"]), rtol=0, atol=1e-14)


# ---------------------------------------------------------------- brute force

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_matches_brute_force_tiny(dtype):
    w = W.tiny_decode(0, dtype)
    o, l = oracle.decode(w)
    bo, bl = brute_decode(w)
    np.testing.assert_allclose(o, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, bl, rtol=0, atol=1e-12)


def test_decode_matches_brute_force_irregular():
    w = _scaled_irregular(3, seq_lens=[0, 1, 17, 40], Hq=6, Hkv=2, d=64, max_pos=300)
    o, l = oracle.decode(w)
    bo, bl = brute_decode(w)
    np.testing.assert_allclose(o, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, bl, rtol=0, atol=1e-12)


def test_prefill_matches_brute_force_irregular():
    w = W.irregular_prefill(4, "f32", kv_lens=[5, 33, 20], q_lens=[5, 7, 1], Hq=4, Hkv=2, d=64, max_pos=300)
    o, l = oracle.prefill(w)
    bo, bl = brute_prefill(w)
    np.testing.assert_allclose(o, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, bl, rtol=0, atol=1e-12)


# ---------------------------------------------------------------- equivalences

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_equals_attention_over_private_prerotated_copies(dtype):
    w = W.tiny_decode(0, dtype)
    o, l = oracle.decode(w)
    for r in range(w.decode.batch):
        po, pl = _private_prerotated_decode(w, r)
        np.testing.assert_allclose(o[r], po, rtol=0, atol=1e-12)
        np.testing.assert_allclose(l[r], pl, rtol=0, atol=1e-12)


def test_shared_block_at_different_offsets_and_negative_control():
    w = W.tiny_decode(0, "f32")
    bt, st = w.decode.block_tables, w.decode.block_starts
    shared = [(int(p), int(st[0, i]), int(st[1, list(bt[1]).index(p)]))
              for i, p in enumerate(bt[0]) if p in bt[1]]
    diff = [s for s in shared if s[1] != s[2]]
    assert diff, "workload must share a block at different offsets"
    phys, off0, off1 = diff[0]
    o, _ = oracle.decode(w)
    # reuse the block rotated once at request 0's offset inside request 1
    bad, _ = _private_prerotated_decode(w, 1, shared_override=(phys, off0))
    assert np.max(np.abs(bad - o[1])) > 1e-3


@pytest.mark.parametrize("shift", [1, 4096, 123457])
def test_relative_position_invariant(shift):
    w = _scaled_irregular(5, seq_lens=[33, 100, 7], Hq=4, Hkv=2, d=128, max_pos=8192)
    o, l = oracle.decode(w)
    w.decode.block_starts = w.decode.block_starts + shift
    w.decode.q_pos = w.decode.q_pos + shift
    o2, l2 = oracle.decode(w)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l2, l, rtol=0, atol=1e-12)
    wp = W.irregular_prefill(6, "f32", kv_lens=[40, 9], q_lens=[8, 9], Hq=4, Hkv=1, d=64, max_pos=8192)
    o, l = oracle.prefill(wp)
    wp.prefill.block_starts = wp.prefill.block_starts + shift
    wp.prefill.q_pos = wp.prefill.q_pos + shift
    o2, l2 = oracle.prefill(wp)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-12)


def test_zero_positions_reduce_to_plain_attention():
    # block size 1 so that every key position can be 0
    rng = np.random.default_rng(7)
    L, d, Hq, Hkv = 37, 64, 4, 2
    k = rng.standard_normal((L, Hkv, 1, d)).astype(np.float32)
    v = rng.standard_normal((L, Hkv, 1, d)).astype(np.float32)
    q = rng.standard_normal((1, Hq, d)).astype(np.float32)
    perm = rng.permutation(L).astype(np.int32)
    w = W.Workload("zero", "f32", Hq, Hkv, d, 1, 10000.0, 1, W.PagedKV(k, v))
    w.decode = W.DecodeBatch(q, perm[None, :], np.zeros((1, L), np.int32),
                             np.array([L], np.int32), np.array([0], np.int32))
    o, l = oracle.decode(w)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        K = k[perm, g, 0].astype(np.float64)
        V = v[perm, g, 0].astype(np.float64)
        s = K @ q[0, h].astype(np.float64) / math.sqrt(d)
        np.testing.assert_allclose(o[0, h], softmax(s) @ V, atol=1e-13)
        assert abs(l[0, h] - logsumexp(s)) < 1e-13


# ---------------------------------------------------------------- index pins

def test_single_key_gives_value_row_exactly_and_zero_query_gives_mean():
    w = _scaled_irregular(8, seq_lens=[1, 50, 0], Hq=4, Hkv=2, d=128, max_pos=1000)
    o, l = oracle.decode(w)
    dec = w.decode
    for h in range(w.Hq):
        g = h // 2
        assert np.array_equal(o[0, h], w.kv.v_pool[dec.block_tables[0, 0], g, 0].astype(np.float64))
    assert np.all(o[2] == 0.0) and np.all(np.isneginf(l[2]))
    dec.q[1] = 0.0
    o, l = oracle.decode(w)
    phys, slot, _ = oracle.key_index_map(dec.block_tables[1], dec.block_starts[1], 50, 16)
    for h in range(w.Hq):
        mean = w.kv.v_pool[phys, h // 2, slot].astype(np.float64).mean(axis=0)
        np.testing.assert_allclose(o[1, h], mean, atol=1e-14)
        assert abs(l[1, h] - math.log(50)) < 1e-14


def test_output_in_convex_hull_and_lse():
    w = W.tiny_decode(1, "f32")
    o, l = oracle.decode(w)
    dec = w.decode
    for r in range(dec.batch):
        for h in range(w.Hq):
            phys, slot, _ = oracle.key_index_map(dec.block_tables[r], dec.block_starts[r], int(dec.seq_lens[r]), 16)
            V = w.kv.v_pool[phys, h // 2, slot].astype(np.float64)
            assert np.all(o[r, h] <= V.max(axis=0) + 1e-12) and np.all(o[r, h] >= V.min(axis=0) - 1e-12)
            assert l[r, h] > -1e9


def test_prefill_rows_equal_decode_with_key_prefix():
    wp = W.irregular_prefill(9, "f32", kv_lens=[45, 16], q_lens=[12, 16], Hq=4, Hkv=2, d=64, max_pos=2048)
    o, l = oracle.prefill(wp)
    pre = wp.prefill
    for r in range(pre.batch):
        q0, q1 = int(pre.cu_q_lens[r]), int(pre.cu_q_lens[r + 1])
        ql, kv = q1 - q0, int(pre.kv_lens[r])
        for i in range(ql):
            wd = W.Workload("row", "f32", wp.Hq, wp.Hkv, wp.d, 16, wp.rope_base, wp.max_pos, wp.kv)
            wd.decode = W.DecodeBatch(pre.q[q0 + i][None], pre.block_tables[r][None], pre.block_starts[r][None],
                                      np.array([kv - ql + i + 1], np.int32), np.array([pre.q_pos[q0 + i]], np.int32))
            od, ld = oracle.decode(wd)
            np.testing.assert_allclose(o[q0 + i], od[0], atol=1e-13)
            np.testing.assert_allclose(l[q0 + i], ld[0], atol=1e-13)


def test_index_causality_equals_position_causality_on_workloads():
    """On the RAG workloads positions increase with key index, so the
    by-index causal rule equals 'key position <= query position'."""
    for w in (W.rag_prefill(0, B=2, n_spans=2, span_tokens=256, pool_spans=8, q_len=64),
              W.mixed_batch(0, n_prefill=2, chunk=128, n_decode=2, min_ctx=64, max_ctx=300)):
        pre = w.prefill
        for r in range(pre.batch):
            q0, q1 = int(pre.cu_q_lens[r]), int(pre.cu_q_lens[r + 1])
            ql, kv = q1 - q0, int(pre.kv_lens[r])
            _, _, pos = oracle.key_index_map(pre.block_tables[r], pre.block_starts[r], kv, 16)
            for i in range(ql):
                by_index = np.arange(kv) <= kv - ql + i
                by_pos = pos <= pre.q_pos[q0 + i]
                assert np.array_equal(by_index, by_pos)


# ---------------------------------------------------------------- planted mistakes

def _mut_sign(x, pos, base):
    x = np.asarray(x, np.float64)
    h = x.shape[-1] // 2
    c, s = oracle.rope_cos_sin(pos, x.shape[-1], base)
    out = np.empty_like(x)
    out[..., :h] = x[..., :h] * c + x[..., h:] * s
    out[..., h:] = x[..., h:] * c - x[..., :h] * s
    return out


def _mut_interleaved(x, pos, base):
    x = np.asarray(x, np.float64)
    c, s = oracle.rope_cos_sin(pos, x.shape[-1], base)
    out = np.empty_like(x)
    out[..., 0::2] = x[..., 0::2] * c - x[..., 1::2] * s
    out[..., 1::2] = x[..., 1::2] * c + x[..., 0::2] * s
    return out


def _mut_freq(x, pos, base):
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    h = d // 2
    ang = np.asarray(pos, np.float64)[:, None] * (base ** (-np.arange(h) / d))[None, :]
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(x)
    out[..., :h] = x[..., :h] * c - x[..., h:] * s
    out[..., h:] = x[..., h:] * c + x[..., :h] * s
    return out


def _mut_keypos(table_row, start_row, n_keys, bs):
    phys, slot, pos = _orig_key_index_map(table_row, start_row, n_keys, bs)
    return phys, slot, pos + 1


_orig_key_index_map = oatt.key_index_map


def _pins_pass():
    """Run a compact set of the pins above; return True if all hold."""
    try:
        for c in json.load(open(GOLDEN))["cases"]:
            test_worked_examples(c)
        w = W.tiny_decode(0, "f32")
        o, l = oracle.decode(w)
        bo, bl = brute_decode(w)
        if np.max(np.abs(o - bo)) > 1e-12:
            return False
        for r in range(2):
            po, _ = _private_prerotated_decode(w, r)
            if np.max(np.abs(o[r] - po)) > 1e-12:
                return False
        test_table_closed_forms(64, 10000.0)
    except AssertionError:
        return False
    return True


@pytest.mark.parametrize("where,mutant", [
    ("rope_rotate", _mut_sign),
    ("rope_rotate", _mut_interleaved),
    ("rope_rotate", _mut_freq),
    ("key_index_map", _mut_keypos),
])
def test_pins_catch_planted_mistakes(monkeypatch, where, mutant):
    assert _pins_pass()
    monkeypatch.setattr(oatt, where, mutant)
    if where == "rope_rotate":
        monkeypatch.setattr(oracle, "rope_rotate", mutant)
    assert not _pins_pass()


def test_pins_catch_wrong_gqa_mapping(monkeypatch):
    def bad_decode(w, requests=None, scale=0.0):
        dec = w.decode
        out = np.zeros((dec.batch, w.Hq, w.d))
        lse = np.zeros((dec.batch, w.Hq))
        for r in range(dec.batch):
            for h in range(w.Hq):
                # wrong: head h reads kv head h % Hkv instead of h // G
                k, v, pos = oatt._gathered(w, dec.block_tables[r], dec.block_starts[r], int(dec.seq_lens[r]),
                                           h % w.Hkv)
                qr = oracle.rope_rotate(oracle.widen(dec.q[r, h][None, :], w.dtype), [int(dec.q_pos[r])],
                                        w.rope_base)
                o, l = oracle.attend(qr, oracle.rope_rotate(k, pos, w.rope_base), v, 1.0 / np.sqrt(w.d))
                out[r, h], lse[r, h] = o[0], l[0]
        return out, lse
    w = W.tiny_decode(0, "f32")
    bo, _ = brute_decode(w)
    assert np.max(np.abs(oracle.decode(w)[0] - bo)) < 1e-12
    assert np.max(np.abs(bad_decode(w)[0] - bo)) > 1e-3
