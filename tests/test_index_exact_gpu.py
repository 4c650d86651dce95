"""Exact indexing on the GPU, through the C ABI.

Which (physical block, slot) pairs each kernel gathers for each query row,
and, for the fp32 decode, the logical position pi(j) = start[r][j / 16] + j % 16
at which it rotates every key, are read back from the outputs as integer
counts (value rows carry codes, see ``index_codes``) and compared with the
counts of the oracle's output and with the counts taken directly from the
oracle's key index map: integers, compared with ``np.array_equal``.
(MiniPIC summary, section 2.1: pi(j) is the logical position of stored key j
inside the current request; one physical block may serve several requests, and
several offsets of one request, at once.)
"""

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import i32, to_dev, upload_decode, upload_prefill
from index_codes import (ALIGNED, aligned_decode, coded_values, counts, counts_from_indices, phase_margin,
                         zero_query_decode, zero_query_prefill)

pytestmark = pytest.mark.gpu

# How far n * out may sit from the exact count c: fp32 outputs carry ~1e-7
# relative error, bf16 outputs a rounding of at most 2^-9 relative (plus the
# fp32 sums before it).  Counts are kept below 110 in the bf16 cases, so the
# bound stays under 1/2 and the nearest integer is the count.
def _tol(c, dtype):
    return 1e-3 + 0.0 * c if dtype == "f32" else 2.0 ** -8 * c + 0.05


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


def _decode_gpu(env, w):
    torch, mp, dev = env
    t = upload_decode(w, torch, dev)
    rope = mp.rope_table(w.max_pos, w.d, w.rope_base, device=dev)
    lse = torch.full((w.decode.batch, w.Hq), float("nan"), dtype=torch.float32, device=dev)
    out, _ = mp.attn_decode(t["q"], t["k_pool"], t["v_pool"], t["block_tables"], t["block_starts"],
                            t["seq_lens"], t["q_pos"], rope, lse=lse)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


def _prefill_gpu(env, w):
    torch, mp, dev = env
    p = w.prefill
    t = upload_prefill(w, torch, dev)
    rope = mp.rope_table(w.max_pos, w.d, w.rope_base, device=dev)
    out, _ = mp.attn_prefill(t["q"], t["cu_q_lens"], t["q_pos"], t["k_pool"], t["v_pool"], t["block_tables"],
                             t["block_starts"], t["kv_lens"], rope, max_q_len=int(np.diff(p.cu_q_lens).max()))
    torch.cuda.synchronize()
    return out.float().cpu().numpy()


def _check_row(got, ref, phys, slot, n, g, dtype, what):
    """One query row: the GPU's counts equal the oracle's and the index map's."""
    d = got.shape[-1]
    if n == 0:
        assert np.all(got == 0.0), what
        return
    cg, _ = counts(got, n)
    cr, fr = counts(ref, n)
    assert fr < 1e-4, f"{what}: oracle counts not integral ({fr})"
    exp = counts_from_indices(phys, slot, d)
    tol = _tol(exp, dtype)
    assert np.all(tol < 0.5), f"{what}: counts too large to resolve in {dtype}"
    assert np.array_equal(cr, exp), f"{what}: oracle counts differ from its index map"
    assert np.array_equal(cg, exp), f"{what}: gathered set differs: {np.nonzero(cg != exp)[0]}"
    x = np.asarray(got[:-1], dtype=np.float64) * n
    assert np.all(np.abs(x - exp) <= tol), f"{what}: counts off by {np.abs(x - exp).max()}"
    assert abs(got[-1] - (g + 1)) <= 1e-5 * (g + 1) + (2.0 ** -8 if dtype == "bf16" else 0.0), f"{what}: kv head"


def _decode_counts_equal(w, out, ref):
    dec = w.decode
    G = w.Hq // w.Hkv
    for r in range(dec.batch):
        n = int(dec.seq_lens[r])
        phys, slot, _ = oracle.key_index_map(dec.block_tables[r], dec.block_starts[r], n, w.block_size)
        for h in range(w.Hq):
            _check_row(out[r, h], ref[r, h], phys, slot, n, h // G, w.dtype, f"decode r={r} h={h}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("Hq,Hkv,d", [(8, 2, 128), (6, 2, 64), (28, 4, 128), (16, 1, 64)])
def test_decode_gathers_exactly_the_oracles_keys(env, dtype, Hq, Hkv, d):
    """q = 0: every key of a request weighs 1/n, so n * out counts the
    (block, slot) pairs gathered; random block ids (repeated within and across
    requests) and random starts."""
    w = zero_query_decode(40 + Hq + d, dtype, Hq, Hkv, d, [0, 1, 15, 16, 17, 100, 250, 700, 1000])
    out, lse = _decode_gpu(env, w)
    ref, _ = oracle.decode(w)
    _decode_counts_equal(w, out, ref)
    assert env[1].device_error() == 0


def test_decode_gathers_exactly_in_a_large_batch(env):
    """The same with enough requests that the grid spans several waves and
    splits of different lengths."""
    rng = np.random.default_rng(7)
    lens = rng.integers(0, 1500, size=96).tolist()
    w = zero_query_decode(41, "bf16", 32, 8, 128, lens)
    out, _ = _decode_gpu(env, w)
    ref, _ = oracle.decode(w)
    _decode_counts_equal(w, out, ref)


@pytest.mark.parametrize("Hq,Hkv,d", [(8, 2, 128), (32, 8, 128), (7, 1, 128), (12, 4, 64), (4, 4, 64)])
def test_prefill_gathers_exactly_the_oracles_keys(env, Hq, Hkv, d):
    """q = 0: chunk query i of request r weighs the keys j <= kv - q_len + i
    equally; the counts of every row equal the oracle's, over ragged chunks
    that span several key tiles."""
    w = zero_query_prefill(50 + Hq + d, Hq, Hkv, d, kv_lens=[1, 17, 300, 129, 513, 700, 40],
                           q_lens=[1, 5, 300, 1, 77, 160, 0])
    out = _prefill_gpu(env, w)
    ref, _ = oracle.prefill(w)
    p = w.prefill
    G = Hq // Hkv
    for r in range(p.batch):
        q0, q1 = int(p.cu_q_lens[r]), int(p.cu_q_lens[r + 1])
        kv = int(p.kv_lens[r])
        phys_all, slot_all, _ = oracle.key_index_map(p.block_tables[r], p.block_starts[r], kv, 16)
        for i in range(q1 - q0):
            n = kv - (q1 - q0) + i + 1
            for h in range(Hq):
                _check_row(out[q0 + i, h], ref[q0 + i, h], phys_all[:n], slot_all[:n], n, h // G, "bf16",
                           f"prefill r={r} i={i} h={h}")
    assert env[1].device_error() == 0


def test_mixed_launch_gathers_exactly_the_oracles_keys(env):
    """Prefill chunks and decode tokens in one launch over one coded pool."""
    torch, mp, dev = env
    d, Hq, Hkv = 128, 16, 2
    wp = W.irregular_prefill(60, "bf16", kv_lens=[300, 513, 90], q_lens=[300, 77, 90], Hq=Hq, Hkv=Hkv, d=d,
                             max_pos=60000, pool_blocks=d - 17)
    wd = W.irregular_decode(61, "bf16", seq_lens=[0, 1, 33, 700, 1500], Hq=Hq, Hkv=Hkv, d=d, max_pos=60000,
                            pool_blocks=d - 17)
    wp.prefill.q[:] = 0
    wd.decode.q[:] = 0
    wp.kv.v_pool = coded_values(wp.kv.num_blocks, Hkv, 16, d, "bf16")
    wd.kv = wp.kv
    p, dd = wp.prefill, wd.decode
    kpool, vpool = to_dev(wp.kv.k_pool, "bf16", torch, dev), to_dev(wp.kv.v_pool, "bf16", torch, dev)
    rope = mp.rope_table(60000, d, wp.rope_base, device=dev)
    pre = dict(q=to_dev(p.q, "bf16", torch, dev), cu_q_lens=i32(p.cu_q_lens, torch, dev),
               q_pos=i32(p.q_pos, torch, dev), block_tables=i32(p.block_tables, torch, dev),
               block_starts=i32(p.block_starts, torch, dev), kv_lens=i32(p.kv_lens, torch, dev),
               max_q_len=int(np.diff(p.cu_q_lens).max()))
    dec = dict(q=to_dev(dd.q, "bf16", torch, dev), block_tables=i32(dd.block_tables, torch, dev),
               block_starts=i32(dd.block_starts, torch, dev), seq_lens=i32(dd.seq_lens, torch, dev),
               q_pos=i32(dd.q_pos, torch, dev))
    po, _, do, _ = mp.attn_mixed(pre, dec, kpool, vpool, rope)
    torch.cuda.synchronize()
    po, do = po.float().cpu().numpy(), do.float().cpu().numpy()
    _decode_counts_equal(wd, do, oracle.decode(wd)[0])
    ref, _ = oracle.prefill(wp)
    G = Hq // Hkv
    for r in range(p.batch):
        q0, q1 = int(p.cu_q_lens[r]), int(p.cu_q_lens[r + 1])
        kv = int(p.kv_lens[r])
        phys_all, slot_all, _ = oracle.key_index_map(p.block_tables[r], p.block_starts[r], kv, 16)
        for i in range(q1 - q0):
            n = kv - (q1 - q0) + i + 1
            for h in range(Hq):
                _check_row(po[q0 + i, h], ref[q0 + i, h], phys_all[:n], slot_all[:n], n, h // G, "bf16",
                           f"mixed prefill r={r} i={i} h={h}")
    assert mp.device_error() == 0


def test_decode_rotates_every_key_at_its_exact_position(env):
    """fp32 decode.  Every key k~_j is stored pre-rotated back by the oracle's
    pi(j), and the query by its position, so that after a correct rotation all
    keys of a (request, kv head) score the same M; a key rotated at any other
    position keeps at most phase_margin * M, i.e. >= 25 less, and drops out of
    the softmax.  The counts then equal the oracle's only if every key was
    rotated at exactly pi(j), and the lse equals M + log n only if the query
    was rotated at exactly its position."""
    c = ALIGNED
    M = c["M"]
    assert M * (1.0 - phase_margin(c["d"], 10000.0, c["n_pairs"], 2 * c["max_pos"])) >= 25.0
    w = aligned_decode()
    out, lse = _decode_gpu(env, w)
    ref, rl = oracle.decode(w)
    _decode_counts_equal(w, out, ref)
    n = np.asarray(c["seq"], dtype=np.float64)[:, None]
    assert np.abs(rl - (M + np.log(n))).max() < 1e-6 * M
    assert np.abs(lse - (M + np.log(n))).max() < 0.05
