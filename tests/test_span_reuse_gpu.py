"""Span reuse end to end: the library's block-hash chain and prefix cache
(MiniPIC summary, section 2.2: SSEP restarts the chain so a span is cached
whatever precedes it; PDEP ties the question to the whole prompt) turn RAG
prompts into block tables and starts, and the GPU decode reads the shared
physical blocks at each request's own offsets (section 2.1).  Checked against
the oracle on the same tables."""

import numpy as np
import pytest

import oracle
import workloads as W
from gpu_util import compare, compare_lse, upload_decode

pytestmark = pytest.mark.gpu

SSEP, PDEP = 128001, 128002
BS = 16


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


def _prompts(rng, n_req, n_spans_pool, spans_per_req):
    spans = []
    for _ in range(n_spans_pool):
        nb = int(rng.integers(1, 5))
        spans.append([SSEP] + list(rng.integers(0, 100000, size=nb * BS - 1)))
    system = list(rng.integers(0, 100000, size=2 * BS))
    prompts = []
    for _ in range(n_req):
        toks = list(system)
        for s in rng.choice(n_spans_pool, size=spans_per_req, replace=False):
            toks += spans[s]
        toks += [PDEP] + list(rng.integers(0, 100000, size=int(rng.integers(BS - 1, 3 * BS))))
        prompts.append(toks)
    return prompts


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prefix_cache_tables_drive_the_decode(env, dtype):
    torch, mp, dev = env
    rng = np.random.default_rng(11)
    prompts = _prompts(rng, n_req=12, n_spans_pool=10, spans_per_req=5)
    cache = mp.PrefixCache(4096)
    tabs, starts = [], []
    for p in prompts:
        n_blocks = -(-len(p) // BS)
        t, s, _ = cache.assign(mp.block_hashes(p, BS, SSEP, PDEP), n_blocks, BS)
        tabs.append(np.asarray(t))
        starts.append(np.asarray(s))
    # blocks are shared across requests, and some shared block sits at different
    # logical starts in two requests
    where = {}
    for r, (t, s) in enumerate(zip(tabs, starts)):
        for blk, st in zip(t, s):
            where.setdefault(int(blk), set()).add(int(st))
    assert any(len(v) > 1 for v in where.values())
    B, Hq, Hkv, d = len(prompts), 16, 4, 128
    mb = max(len(t) for t in tabs)
    bt = np.zeros((B, mb), dtype=np.int32)
    st = np.zeros((B, mb), dtype=np.int32)
    for r in range(B):
        bt[r, :len(tabs[r])] = tabs[r]
        st[r, :len(starts[r])] = starts[r]
    seq = np.array([len(p) for p in prompts], dtype=np.int32)
    nblk = int(bt.max()) + 1
    k = rng.standard_normal((nblk, Hkv, BS, d)).astype(np.float32)
    v = rng.standard_normal((nblk, Hkv, BS, d)).astype(np.float32)
    q = rng.standard_normal((B, Hq, d)).astype(np.float32)
    if dtype == "bf16":
        k, v, q = W.to_bf16_bits(k), W.to_bf16_bits(v), W.to_bf16_bits(q)
    max_pos = int(seq.max()) + 1
    w = W.Workload("span_reuse", dtype, Hq, Hkv, d, BS, 500000.0, max_pos, W.PagedKV(k, v),
                   decode=W.DecodeBatch(q, bt, st, seq, seq.copy()))
    t = upload_decode(w, torch, dev)
    rope = mp.rope_table(max_pos, d, w.rope_base, device=dev)
    lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev)
    out, _ = mp.attn_decode(t["q"], t["k_pool"], t["v_pool"], t["block_tables"], t["block_starts"],
                            t["seq_lens"], t["q_pos"], rope, lse=lse)
    torch.cuda.synchronize()
    ref, rl = oracle.decode(w)
    compare(out.float().cpu().numpy(), ref, dtype, "decode over prefix-cache tables")
    compare_lse(lse.cpu().numpy(), rl, dtype, "decode over prefix-cache tables")
    assert mp.device_error() == 0
