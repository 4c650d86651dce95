"""Decode parity: the CUDA path (through the C ABI) against the CPU oracle."""

import os

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import TOL, compare, compare_lse, upload_decode, to_dev, i32
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


def run_decode(env, w, prerotated=False, t=None, rope=None):
    torch, mp, dev = env
    t = t or upload_decode(w, torch, dev)
    lse = torch.full((w.decode.batch, w.Hq), float("nan"), dtype=torch.float32, device=dev)
    if prerotated:
        out, _ = mp.attn_decode_prerotated(t["q"], t["k_pool"], t["v_pool"], t["block_tables"],
                                           t["block_starts"], t["seq_lens"], t["q_pos"], lse=lse)
    else:
        rope = rope if rope is not None else mp.rope_table(w.max_pos, w.d, w.rope_base, device=dev)
        out, _ = mp.attn_decode(t["q"], t["k_pool"], t["v_pool"], t["block_tables"], t["block_starts"],
                                t["seq_lens"], t["q_pos"], rope, lse=lse)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("d,base,max_pos", [(64, 10000.0, 129), (128, 500000.0, 131073), (128, 1e6, 32769)])
def test_rope_table_within_one_ulp(env, d, base, max_pos):
    torch, mp, dev = env
    T = mp.rope_table(max_pos, d, base, device=dev).cos_sin.cpu().numpy().astype(np.float64)
    R = oracle.rope_table(max_pos, d, base)
    ulp = np.spacing(np.abs(R).astype(np.float32)).astype(np.float64)
    # the fp64 angle p*theta carries an absolute error of a few ulp(p*theta) <= ~6e-11;
    # next to zero that is many fp32 ulps, elsewhere the bound is one fp32 ulp
    angle_err = 8 * max_pos * 2.0 ** -52
    assert np.all(np.abs(T - R) <= ulp + angle_err)


@pytest.mark.parametrize("d,base,max_pos", [(64, 10000.0, 129), (128, 500000.0, 131073), (128, 1e6, 32769)])
def test_rope_table_f16_rounds_once_to_nearest(env, d, base, max_pos):
    """The fp16 table is the exact value rounded once to the nearest fp16: within
    half an fp16 spacing of the oracle's float64 value (spacing 2^-24 below
    2^-14, where fp16 numbers are subnormal), plus the fp64 angle error; and its
    fp16 neighbours are not closer."""
    torch, mp, dev = env
    T = mp.rope_table(max_pos, d, base, device=dev).cos_sin_f16.cpu().numpy()
    R = oracle.rope_table(max_pos, d, base)
    Th = T.astype(np.float64)
    spacing = np.spacing(np.abs(Th).astype(np.float16)).astype(np.float64)
    angle_err = 8 * max_pos * 2.0 ** -52
    assert np.all(np.abs(Th - R) <= 0.5 * spacing + angle_err)
    assert np.all(np.isfinite(Th)) and np.all(np.abs(Th) <= 1.0)


@pytest.mark.parametrize("d,base,max_pos", [(64, 10000.0, 129), (128, 500000.0, 131073), (128, 1e6, 32769)])
def test_rope_table_bf16_rows(env, d, base, max_pos):
    """Rows [p, 0] and [p, 1] of the bf16 table are cos | sin | -sin of +p theta_i
    and of -p theta_i: each value the fp32 table's value rounded to the nearest
    bf16 (so within half a bf16 spacing plus one fp32 ulp and the fp64 angle
    error of the oracle), with the signs placed exactly."""
    torch, mp, dev = env
    tab = mp.rope_table(max_pos, d, base, device=dev)
    B = tab.cos_sin_bf16
    assert tuple(B.shape) == (max_pos, 2, 3 * d // 2)
    h = d // 2
    # round to nearest even of the fp32 table (torch's conversion, not the kernel's)
    c = tab.cos_sin[:, :h].to(torch.bfloat16)
    s = tab.cos_sin[:, h:].to(torch.bfloat16)
    assert torch.equal(B[:, 0, :h], c) and torch.equal(B[:, 1, :h], c)
    assert torch.equal(B[:, 0, h:2 * h], s) and torch.equal(B[:, 0, 2 * h:], -s)
    assert torch.equal(B[:, 1, h:2 * h], -s) and torch.equal(B[:, 1, 2 * h:], s)
    R = oracle.rope_table(max_pos, d, base)
    Bf = B[:, 0].float().cpu().numpy().astype(np.float64)
    got = np.concatenate([Bf[:, :h], Bf[:, h:2 * h]], axis=1)
    ulp32 = np.spacing(np.abs(R).astype(np.float32)).astype(np.float64)
    half_bf16 = np.ldexp(1.0, np.frexp(np.abs(got))[1] - 9)  # half a bf16 spacing at |got|
    angle_err = 8 * max_pos * 2.0 ** -52
    assert np.all(np.abs(got - R) <= half_bf16 + ulp32 + angle_err)


def test_rope_tables_one_pass_equals_the_single_forms(env):
    """minipic_rope_tables writes the same bits as the three single-form calls."""
    torch, mp, dev = env
    tab = mp.rope_table(4097, 128, 500000.0, device=dev)
    f32 = torch.empty_like(tab.cos_sin)
    assert mp.load().minipic_rope_table(f32.data_ptr(), 4097, 128, 500000.0, None) == 0
    f16 = mp.rope_table_f16(4097, 128, 500000.0, device=dev)
    b16 = mp.rope_table_bf16(4097, 128, 500000.0, device=dev)
    torch.cuda.synchronize()
    assert torch.equal(f32.view(torch.int32), tab.cos_sin.view(torch.int32))
    assert torch.equal(f16.view(torch.int16), tab.cos_sin_f16.view(torch.int16))
    assert torch.equal(b16.view(torch.int16), tab.cos_sin_bf16.view(torch.int16))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_tiny_decode(env, dtype):
    w = W.tiny_decode(0, dtype)
    out, lse = run_decode(env, w)
    ref, rl = oracle.decode(w)
    compare(out, ref, dtype, "tiny_decode")
    compare_lse(lse, rl, dtype, "tiny_decode")
    assert env[1].device_error() == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rag_decode_scaled(env, dtype):
    w = W.rag_decode(1, dtype, B=3, n_spans=6, span_tokens=256, pool_spans=16, tail_tokens=77)
    out, lse = run_decode(env, w)
    ref, rl = oracle.decode(w)
    compare(out, ref, dtype, "rag_decode small")
    compare_lse(lse, rl, dtype, "rag_decode small")


def test_long_decode_scaled(env):
    w = W.long_decode(2, "bf16", B=2, n_spans=6, span_tokens=4096, pool_spans=5)
    out, lse = run_decode(env, w)
    ref, rl = oracle.decode(w)
    compare(out, ref, "bf16", "long_decode small")
    compare_lse(lse, rl, "bf16", "long_decode small")


def test_mixed_decode_part_scaled(env):
    w = W.mixed_batch(3, n_prefill=0, n_decode=6, min_ctx=1, max_ctx=3000)
    out, lse = run_decode(env, w)
    ref, rl = oracle.decode(w)
    compare(out, ref, "bf16", "mixed decodes")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("Hq,Hkv,d", [(8, 8, 128), (6, 2, 64), (28, 4, 128), (32, 2, 128), (16, 1, 64)])
def test_irregular_positions_ragged_lengths(env, dtype, Hq, Hkv, d):
    w = W.irregular_decode(11 + Hq, dtype, seq_lens=[0, 1, 15, 16, 17, 250, 1000], Hq=Hq, Hkv=Hkv, d=d,
                           max_pos=70000)
    out, lse = run_decode(env, w)
    ref, rl = oracle.decode(w)
    compare(out, ref, dtype, f"irregular {Hq}/{Hkv}/{d}")
    compare_lse(lse, rl, dtype, "irregular")
    assert np.all(out[0] == 0.0) and np.all(np.isneginf(lse[0]))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_single_key_returns_value_row_bit_exact(env, dtype):
    w = W.irregular_decode(21, dtype, seq_lens=[1] * 9, Hq=8, Hkv=2, d=128, max_pos=100000)
    out, _ = run_decode(env, w)
    dec = w.decode
    for r in range(dec.batch):
        for h in range(w.Hq):
            row = w.kv.v_pool[dec.block_tables[r, 0], h // 4, 0]
            exp = W.bf16_bits_to_f32(row) if dtype == "bf16" else row
            assert np.array_equal(out[r, h].astype(np.float32), exp)


def test_zero_query_gives_mean_of_gathered_values(env):
    w = W.irregular_decode(22, "f32", seq_lens=[37, 300], Hq=4, Hkv=2, d=128, max_pos=5000)
    w.decode.q[:] = 0.0
    out, lse = run_decode(env, w)
    dec = w.decode
    for r in range(dec.batch):
        phys, slot, _ = oracle.key_index_map(dec.block_tables[r], dec.block_starts[r], int(dec.seq_lens[r]), 16)
        for h in range(w.Hq):
            mean = w.kv.v_pool[phys, h // 2, slot].astype(np.float64).mean(0)
            assert np.abs(out[r, h] - mean).max() < 1e-5
            assert abs(lse[r, h] - np.log(dec.seq_lens[r])) < 1e-5


def test_split_invariance(env):
    """A request decoded alone (many splits) equals the same request inside a
    large batch (fewer splits)."""
    w = W.long_decode(4, "bf16", B=24, n_spans=1, span_tokens=4096, pool_spans=3)
    out_b, _ = run_decode(env, w)
    w1 = W.long_decode(4, "bf16", B=24, n_spans=1, span_tokens=4096, pool_spans=3)
    d = w1.decode
    w1.decode = W.DecodeBatch(d.q[:1], d.block_tables[:1], d.block_starts[:1], d.seq_lens[:1], d.q_pos[:1])
    out_1, _ = run_decode(env, w1)
    assert np.abs(out_1[0] - out_b[0]).max() <= 2e-3


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prerotated_variant_equals_oracle_on_private_copies(env, dtype):
    """The rotation-free kernel over a cache pre-rotated on the host (each
    block used at one offset only) equals the oracle over the unrotated cache."""
    w = W.rag_decode(5, dtype, B=3, n_spans=4, span_tokens=128, pool_spans=8, tail_tokens=40, share=False)
    ref, rl = oracle.decode(w)
    dec = w.decode
    k = oracle.widen(w.kv.k_pool, dtype).copy()
    for r in range(dec.batch):
        phys, slot, pos = oracle.key_index_map(dec.block_tables[r], dec.block_starts[r], int(dec.seq_lens[r]), 16)
        for g in range(w.Hkv):
            k[phys, g, slot] = oracle.rope_rotate(k[phys, g, slot], pos, w.rope_base)
    q = np.stack([oracle.rope_rotate(oracle.widen(dec.q[r], dtype), [int(dec.q_pos[r])] * w.Hq, w.rope_base)
                  for r in range(dec.batch)])
    store = (lambda a: W.to_bf16_bits(a.astype(np.float32))) if dtype == "bf16" else (lambda a: a.astype(np.float32))
    w.kv.k_pool = store(k)
    w.decode.q = store(q)
    out, lse = run_decode(env, w, prerotated=True)
    compare(out, ref, dtype, "prerotated")


def test_device_checks_flag_bad_block_ids_and_positions(env):
    torch, mp, dev = env
    w = W.irregular_decode(30, "bf16", seq_lens=[40, 40, 40], Hq=4, Hkv=2, d=128, max_pos=1000)
    mp.device_error(clear=True)
    w.decode.block_tables[0, 1] = w.kv.k_pool.shape[0] + 5    # block id past the pool
    run_decode(env, w)
    assert mp.device_error(clear=True) & 1
    w = W.irregular_decode(30, "bf16", seq_lens=[40, 40, 40], Hq=4, Hkv=2, d=128, max_pos=1000)
    w.decode.block_starts[1, 0] = 5000                          # position past the table
    run_decode(env, w)
    assert mp.device_error(clear=True) & 2
    w = W.irregular_decode(30, "bf16", seq_lens=[40, 40, 40], Hq=4, Hkv=2, d=128, max_pos=1000)
    w.decode.seq_lens[2] = 10 ** 6                              # longer than the table row
    run_decode(env, w)
    assert mp.device_error(clear=True) & 4
    assert mp.device_error(clear=True) == 0


# ---------------------------------------------------------------- full sizes (sampled outputs)

@pytest.mark.parametrize("idx,sample", [(1, list(range(64))), (3, list(range(8))), (4, list(range(0, 128, 2)))])
def test_full_size_decode(env, idx, sample):
    """The full workloads in the bench's launch configuration: all 64 RAG
    requests, all 8 long-context requests, 64 of the mixed batch's 128
    decodes, each against the oracle (run on every host core)."""
    torch, mp, dev = env
    w = W.config(idx)
    if idx == 4:
        w.prefill = None
    out, lse = run_decode(env, w)
    with OraclePool(w, n_workers=min(len(sample), os.cpu_count() or 1)) as op:
        ref, rl = op.decode(sample)
    compare(out[sample], ref[sample], "bf16", f"config {idx} sampled")
    compare_lse(lse[sample], rl[sample], "bf16", f"config {idx} sampled")
    assert np.all(np.isfinite(out))
    assert mp.device_error() == 0
