"""Mixed continuous batch (span prefills + decodes in ONE launch) against the
CPU oracle, and against the standalone prefill and decode calls."""

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import compare, compare_lse, i32, to_dev
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


def run_mixed(env, w):
    torch, mp, dev = env
    p, d = w.prefill, w.decode
    kpool, vpool = to_dev(w.kv.k_pool, "bf16", torch, dev), to_dev(w.kv.v_pool, "bf16", torch, dev)
    rope = mp.rope_table(w.max_pos, w.d, w.rope_base, device=dev)
    pre = dict(q=to_dev(p.q, "bf16", torch, dev), cu_q_lens=i32(p.cu_q_lens, torch, dev),
               q_pos=i32(p.q_pos, torch, dev), block_tables=i32(p.block_tables, torch, dev),
               block_starts=i32(p.block_starts, torch, dev), kv_lens=i32(p.kv_lens, torch, dev),
               max_q_len=int(np.diff(p.cu_q_lens).max()),
               lse=torch.full((int(p.cu_q_lens[-1]), w.Hq), float("nan"), device=dev))
    dec = dict(q=to_dev(d.q, "bf16", torch, dev), block_tables=i32(d.block_tables, torch, dev),
               block_starts=i32(d.block_starts, torch, dev), seq_lens=i32(d.seq_lens, torch, dev),
               q_pos=i32(d.q_pos, torch, dev), lse=torch.full((d.batch, w.Hq), float("nan"), device=dev))
    po, pl, do, dl = mp.attn_mixed(pre, dec, kpool, vpool, rope)
    torch.cuda.synchronize()
    return (po.float().cpu().numpy(), pl.cpu().numpy(), do.float().cpu().numpy(), dl.cpu().numpy(),
            (pre, dec, kpool, vpool, rope))


def test_mixed_scaled_matches_oracle(env):
    w = W.mixed_batch(5, n_prefill=3, chunk=300, n_decode=6, min_ctx=1, max_ctx=5000)
    po, pl, do, dl, _ = run_mixed(env, w)
    rp, rpl = oracle.prefill(w)
    rd, rdl = oracle.decode(w)
    compare(po, rp, "bf16", "mixed prefill part")
    compare_lse(pl, rpl, "bf16", "mixed prefill part")
    compare(do, rd, "bf16", "mixed decode part")
    compare_lse(dl, rdl, "bf16", "mixed decode part")
    assert env[1].device_error() == 0


def test_mixed_large_groups_match_oracle(env):
    """Groups of 16 query heads per kv head: the decode CTAs of the mixed grid
    take the layout for large groups (two n-tiles, 8 warps with 232 registers)
    and the prefill tiles hold 8 tokens x 16 heads."""
    w = W.mixed_batch(7, n_prefill=2, chunk=200, n_decode=5, min_ctx=1, max_ctx=3000, Hq=32, Hkv=2)
    po, pl, do, dl, _ = run_mixed(env, w)
    rp, rpl = oracle.prefill(w)
    rd, rdl = oracle.decode(w)
    compare(po, rp, "bf16", "mixed prefill part, G 16")
    compare_lse(pl, rpl, "bf16", "mixed prefill part, G 16")
    compare(do, rd, "bf16", "mixed decode part, G 16")
    compare_lse(dl, rdl, "bf16", "mixed decode part, G 16")
    assert env[1].device_error() == 0


def test_mixed_head_dim_64_matches_oracle(env):
    """Head dim 64 runs the single-CTA prefill body with decode CTAs of the same
    shape in one grid."""
    w = W.mixed_batch(8, n_prefill=3, chunk=250, n_decode=7, min_ctx=1, max_ctx=4000, Hq=12, Hkv=4, d=64)
    po, pl, do, dl, _ = run_mixed(env, w)
    rp, rpl = oracle.prefill(w)
    rd, rdl = oracle.decode(w)
    compare(po, rp, "bf16", "mixed d64 prefill part")
    compare(do, rd, "bf16", "mixed d64 decode part")
    compare_lse(dl, rdl, "bf16", "mixed d64 decode part")
    assert env[1].device_error() == 0


def test_mixed_equals_separate_calls(env):
    torch, mp, dev = env
    w = W.mixed_batch(6, n_prefill=2, chunk=200, n_decode=5, min_ctx=100, max_ctx=3000, Hq=16, Hkv=2)
    po, pl, do, dl, (pre, dec, kpool, vpool, rope) = run_mixed(env, w)
    so, _ = mp.attn_prefill(pre["q"], pre["cu_q_lens"], pre["q_pos"], kpool, vpool, pre["block_tables"],
                            pre["block_starts"], pre["kv_lens"], rope, max_q_len=pre["max_q_len"])
    sd, _ = mp.attn_decode(dec["q"], kpool, vpool, dec["block_tables"], dec["block_starts"], dec["seq_lens"],
                           dec["q_pos"], rope)
    torch.cuda.synchronize()
    # for head dim 128 the mixed grid's prefill clusters run the same CTA-pair body
    # as the standalone prefill: the same sums in the same order, bit for bit
    assert np.array_equal(so.float().cpu().numpy(), po)
    # decode CTAs in the mixed grid spread a split over 8 warps instead of 4, which
    # groups the per-warp partial sums differently: equal up to rounding
    diff = np.abs(sd.float().cpu().numpy() - do)
    assert diff.max() <= 4e-3 and diff.mean() <= 2e-4


def test_full_size_mixed(env):
    """The full mixed batch in one launch: 4 of its 16 span prefills and 16 of
    its 128 decodes against the oracle (run on every host core)."""
    w = W.config(4)
    po, pl, do, dl, _ = run_mixed(env, w)
    pre, dec = [0, 5, 10, 15], list(range(3, 128, 8))
    with OraclePool(w) as op:
        rp, rpl = op.prefill(pre)
        rd, rdl = op.decode(dec)
    p = w.prefill
    rows = np.concatenate([np.arange(p.cu_q_lens[r], p.cu_q_lens[r + 1]) for r in pre])
    compare(po[rows], rp[rows], "bf16", "mixed full prefill")
    compare(do[dec], rd[dec], "bf16", "mixed full decode")
    compare_lse(dl[dec], rdl[dec], "bf16", "mixed full decode")
    assert np.all(np.isfinite(po)) and np.all(np.isfinite(do))
    assert env[1].device_error() == 0
