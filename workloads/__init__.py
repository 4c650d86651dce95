"""Seeded synthetic RAG-shaped inputs for position-free paged attention.

This module draws inputs only: span layouts, physical block ids, per-block
logical start positions and N(0,1) values.  It holds none of the attention or
rotary arithmetic, so the CPU oracle and the CUDA path can both read it
without sharing any of the method's computation.

Layout conventions (shared by every consumer):

* ``k_pool`` / ``v_pool``: ``[num_blocks, H_kv, block_size, d]``.  For
  ``dtype == "f32"`` they are ``float32``; for ``dtype == "bf16"`` they hold
  the raw bfloat16 bit patterns as ``uint16``.
* ``block_tables[r][b]``: physical block id of request ``r``'s ``b``-th logical
  block (``int32``; unused entries are -1).
* ``block_starts[r][b]``: logical position of the first token of that block in
  request ``r`` (``int32``).  The key at request-local index ``j`` sits at
  position ``block_starts[r][j // bs] + j % bs``.
* Keys are unrotated.  Queries are unrotated; ``q_pos`` gives their positions.

The five workloads follow the RAG shapes of the MiniPIC summary pages
(gist.science paper 2606.13126, section 4: Llama-3-8B attention shape, retrieved
spans reused at different offsets); every input is synthetic and seeded.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np

BLOCK_SIZE = 16

__all__ = [
    "BLOCK_SIZE",
    "PagedKV",
    "DecodeBatch",
    "PrefillBatch",
    "Workload",
    "to_bf16_bits",
    "bf16_bits_to_f32",
    "build_workload",
    "tiny_decode",
    "rag_decode",
    "rag_prefill",
    "long_decode",
    "mixed_batch",
    "config",
    "CONFIG_NAMES",
]


# ----------------------------------------------------------------------------
# bfloat16 storage helpers (data format only)
# ----------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    bias = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------
# Containers
# ----------------------------------------------------------------------------

@dataclass
class PagedKV:
    k_pool: np.ndarray
    v_pool: np.ndarray

    @property
    def num_blocks(self) -> int:
        return int(self.k_pool.shape[0])


@dataclass
class DecodeBatch:
    q: np.ndarray              # [B, Hq, d]
    block_tables: np.ndarray   # int32 [B, max_blocks]
    block_starts: np.ndarray   # int32 [B, max_blocks]
    seq_lens: np.ndarray       # int32 [B]
    q_pos: np.ndarray          # int32 [B]

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])


@dataclass
class PrefillBatch:
    q: np.ndarray              # [total_q, Hq, d]
    cu_q_lens: np.ndarray      # int32 [B + 1]
    q_pos: np.ndarray          # int32 [total_q]
    kv_lens: np.ndarray        # int32 [B]; includes the chunk's own keys
    block_tables: np.ndarray   # int32 [B, max_blocks]
    block_starts: np.ndarray   # int32 [B, max_blocks]

    @property
    def batch(self) -> int:
        return int(self.kv_lens.shape[0])


@dataclass
class Workload:
    name: str
    dtype: str                 # "f32" or "bf16"
    Hq: int
    Hkv: int
    d: int
    block_size: int
    rope_base: float
    max_pos: int               # table rows needed: every position used is < max_pos
    kv: PagedKV
    decode: Optional[DecodeBatch] = None
    prefill: Optional[PrefillBatch] = None
    notes: str = ""
    # bookkeeping for byte accounting (not used by any computation)
    unique_blocks: int = 0
    meta: dict = field(default_factory=dict)


# ----------------------------------------------------------------------------
# Generic builder
# ----------------------------------------------------------------------------

# A request is described as a list of segments.  A segment is either
#   ("span", span_id, n_tokens)   -- tokens 0..n_tokens-1 of a shared pool span
#   ("own", n_tokens)             -- private tokens of this request
# Segments are laid out back to back; span segments start on a block boundary
# (the pages pad spans to KV-block boundaries, MiniPIC section 2.2 item 1).

Segment = Tuple


def _normal(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """N(0,1) drawn in float32 in row chunks; bf16 workloads keep the bits."""
    shape = tuple(int(s) for s in shape)
    n0 = shape[0]
    inner = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    out = np.empty((n0, inner), dtype=np.uint16 if dtype == "bf16" else np.float32)
    rows = max(1, (1 << 24) // max(inner, 1))
    for s in range(0, n0, rows):
        e = min(n0, s + rows)
        x = rng.standard_normal((e - s, inner), dtype=np.float32)
        out[s:e] = to_bf16_bits(x) if dtype == "bf16" else x
    return out.reshape(shape)


def build_workload(
    name: str,
    seed: int,
    dtype: str,
    Hq: int,
    Hkv: int,
    d: int,
    rope_base: float,
    pool_spans: int,
    span_tokens: int,
    decode_requests: Optional[Sequence[Sequence[Segment]]] = None,
    prefill_requests: Optional[Sequence[Tuple[Sequence[Segment], int]]] = None,
    block_size: int = BLOCK_SIZE,
    rng: Optional[np.random.Generator] = None,
    notes: str = "",
    extra_pool_blocks: int = 0,
) -> Workload:
    """Lay requests out over one shared paged pool and draw the values.

    ``prefill_requests`` entries are ``(segments, q_len)``: the last ``q_len``
    tokens of the request are the query chunk (their own keys are in the
    segments too, as an ``("own", n)`` segment).
    """
    assert dtype in ("f32", "bf16")
    rng = np.random.default_rng(seed) if rng is None else rng
    bs = block_size
    span_blocks = -(-span_tokens // bs)
    decode_requests = list(decode_requests or [])
    prefill_requests = list(prefill_requests or [])

    # logical blocks: pool spans first, then private blocks per request
    n_span_blocks = pool_spans * span_blocks
    private_counts = []
    for segs in decode_requests + [p[0] for p in prefill_requests]:
        private_counts.append(sum(-(-s[1] // bs) for s in segs if s[0] == "own"))
    n_private = int(sum(private_counts))
    num_blocks = n_span_blocks + n_private + extra_pool_blocks
    perm = rng.permutation(num_blocks).astype(np.int64)

    def layout(segs, private_base):
        phys, starts = [], []
        pos = 0
        pb = private_base
        for si, seg in enumerate(segs):
            if seg[0] == "span":
                sid, n = int(seg[1]), int(seg[2])
                assert 0 <= sid < pool_spans and 0 < n <= span_tokens
                for b in range(-(-n // bs)):
                    phys.append(perm[sid * span_blocks + b])
                    starts.append(pos + b * bs)
            elif seg[0] == "own":
                n = int(seg[1])
                for b in range(-(-n // bs)):
                    phys.append(perm[n_span_blocks + pb])
                    starts.append(pos + b * bs)
                    pb += 1
            else:
                raise ValueError(seg)
            pos += -(-n // bs) * bs if si + 1 < len(segs) else n
        ntok = pos
        return phys, starts, ntok, pb

    # A span segment that is not the last one occupies whole blocks (padding);
    # the last segment of a request may end mid-block.
    def table(reqs, private_base):
        rows, lens = [], []
        pb = private_base
        for segs in reqs:
            phys, starts, ntok, pb = layout(segs, pb)
            rows.append((phys, starts))
            lens.append(ntok)
        return rows, lens, pb

    d_rows, d_lens, pb = table(decode_requests, 0)
    p_rows, p_lens, pb = table([p[0] for p in prefill_requests], pb)
    assert pb == n_private

    def pack(rows):
        mb = max([len(r[0]) for r in rows] + [1])
        bt = np.full((len(rows), mb), -1, dtype=np.int32)
        st = np.zeros((len(rows), mb), dtype=np.int32)
        for i, (phys, starts) in enumerate(rows):
            bt[i, : len(phys)] = phys
            st[i, : len(starts)] = starts
        return bt, st

    # values: k pool, v pool, then queries (fixed order)
    kpool = _normal(rng, (num_blocks, Hkv, bs, d), dtype)
    vpool = _normal(rng, (num_blocks, Hkv, bs, d), dtype)

    dec = None
    max_pos = 1
    if decode_requests:
        bt, st = pack(d_rows)
        seq = np.asarray(d_lens, dtype=np.int32)
        qpos = seq.copy()  # the decode token sits at position = context length
        q = _normal(rng, (len(decode_requests), Hq, d), dtype)
        dec = DecodeBatch(q=q, block_tables=bt, block_starts=st, seq_lens=seq, q_pos=qpos)
        max_pos = max(max_pos, int(qpos.max()) + 1)
    pre = None
    if prefill_requests:
        bt, st = pack(p_rows)
        kv_lens = np.asarray(p_lens, dtype=np.int32)
        q_lens = np.asarray([p[1] for p in prefill_requests], dtype=np.int32)
        assert np.all(q_lens <= kv_lens)
        cu = np.zeros(len(q_lens) + 1, dtype=np.int32)
        cu[1:] = np.cumsum(q_lens)
        qpos = np.concatenate(
            [np.arange(kv - ql, kv, dtype=np.int32) for kv, ql in zip(kv_lens, q_lens)]
        ) if len(q_lens) else np.zeros(0, np.int32)
        q = _normal(rng, (int(cu[-1]), Hq, d), dtype)
        pre = PrefillBatch(q=q, cu_q_lens=cu, q_pos=qpos, kv_lens=kv_lens,
                           block_tables=bt, block_starts=st)
        max_pos = max(max_pos, int(kv_lens.max()) + 1)

    used = set()
    for bt in ([dec.block_tables] if dec else []) + ([pre.block_tables] if pre else []):
        used.update(int(x) for x in np.unique(bt) if x >= 0)
    return Workload(
        name=name, dtype=dtype, Hq=Hq, Hkv=Hkv, d=d, block_size=bs,
        rope_base=float(rope_base), max_pos=int(max_pos),
        kv=PagedKV(kpool, vpool), decode=dec, prefill=pre, notes=notes,
        unique_blocks=len(used),
    )


def _zipf_probs(n: int, s: float) -> np.ndarray:
    k = np.arange(1, n + 1, dtype=np.float64)
    p = k ** (-s)
    return p / p.sum()


def _zipf_draw(rng, n_pool: int, m: int, s: float, rank_to_id: np.ndarray,
               replace: bool = False) -> List[int]:
    ranks = rng.choice(n_pool, size=m, replace=replace, p=_zipf_probs(n_pool, s))
    return [int(rank_to_id[r]) for r in ranks]


# ----------------------------------------------------------------------------
# The five workloads (and scaled-down variants for fast parity tests)
# ----------------------------------------------------------------------------

def tiny_decode(seed: int = 0, dtype: str = "f32") -> Workload:
    """Tiny decode: 4/2 heads, d=64, base 1e4; 2 requests x 4 spans x 32 tokens
    drawn from a pool of 6 two-block spans; at least one physical block is read
    by both requests at different logical offsets."""
    rng = np.random.default_rng(seed)
    r0 = [0, 1, 2, 3]
    while True:
        r1 = [int(x) for x in rng.choice(6, size=4, replace=False)]
        if any(s in r1 and r1.index(s) != i for i, s in enumerate(r0)):
            break
    reqs = [[("span", s, 32) for s in r] for r in (r0, r1)]
    w = build_workload("tiny_decode", seed, dtype, Hq=4, Hkv=2, d=64,
                       rope_base=10000.0, pool_spans=6, span_tokens=32,
                       decode_requests=reqs, rng=rng,
                       notes="2 requests x 4 spans x 32 tokens from a pool of 6 spans")
    w.meta["spans"] = [r0, r1]
    return w


def rag_decode(seed: int = 0, dtype: str = "bf16", B: int = 64, Hq: int = 32,
               Hkv: int = 8, d: int = 128, rope_base: float = 500000.0,
               system_tokens: int = 256, n_spans: int = 15, span_tokens: int = 512,
               pool_spans: int = 256, tail_tokens: int = 256, zipf_s: float = 1.1,
               share: bool = True) -> Workload:
    """Decode over RAG contexts: a system prompt shared by every request at
    offset 0, ``n_spans`` retrieved spans drawn Zipf(s) without replacement
    from a shared pool, then a private tail (prior turns + question).

    ``share=False`` gives the no-sharing control: every request gets private
    copies of all its blocks (same shapes, no block read twice)."""
    rng = np.random.default_rng(seed)
    rank_to_id = rng.permutation(pool_spans)
    reqs = []
    for _ in range(B):
        spans = _zipf_draw(rng, pool_spans, n_spans, zipf_s, rank_to_id)
        segs = []
        if share:
            if system_tokens:
                segs.append(("span", pool_spans, system_tokens))  # system prompt span
            segs += [("span", s, span_tokens) for s in spans]
        else:
            ntok = system_tokens + n_spans * span_tokens
            segs.append(("own", ntok))
        if tail_tokens:
            segs.append(("own", tail_tokens))
        reqs.append(segs)
    total_pool = pool_spans + 1 if share else 0
    span_len = max(span_tokens, system_tokens)
    ctx = system_tokens + n_spans * span_tokens + tail_tokens
    return build_workload(
        "rag_decode" if share else "rag_decode_private", seed, dtype, Hq, Hkv, d,
        rope_base, pool_spans=total_pool, span_tokens=span_len,
        decode_requests=reqs, rng=rng,
        notes=f"B={B} ctx={ctx}: {system_tokens} sys + {n_spans}x{span_tokens} "
              f"Zipf({zipf_s}) of {pool_spans} + {tail_tokens} private"
              + ("" if share else " (no sharing)"))


def rag_prefill(seed: int = 0, dtype: str = "bf16", B: int = 8, Hq: int = 32,
                Hkv: int = 8, d: int = 128, rope_base: float = 500000.0,
                n_spans: int = 6, span_tokens: int = 1024, pool_spans: int = 64,
                q_len: int = 512, zipf_s: float = 1.1) -> Workload:
    """Chunked prefill of the final prompt over cached spans: each request's
    ``q_len``-token chunk attends causally to its own keys plus ``n_spans``
    cached spans drawn Zipf(s) from a shared pool (different offsets)."""
    rng = np.random.default_rng(seed)
    rank_to_id = rng.permutation(pool_spans)
    reqs = []
    for _ in range(B):
        spans = _zipf_draw(rng, pool_spans, n_spans, zipf_s, rank_to_id)
        segs = [("span", s, span_tokens) for s in spans] + [("own", q_len)]
        reqs.append((segs, q_len))
    return build_workload(
        "rag_prefill", seed, dtype, Hq, Hkv, d, rope_base,
        pool_spans=pool_spans, span_tokens=span_tokens,
        prefill_requests=reqs, rng=rng,
        notes=f"B={B}, chunk {q_len} over {n_spans}x{span_tokens} Zipf({zipf_s}) of {pool_spans}")


def long_decode(seed: int = 0, dtype: str = "bf16", B: int = 8, Hq: int = 64,
                Hkv: int = 8, d: int = 128, rope_base: float = 500000.0,
                n_spans: int = 32, span_tokens: int = 4096, pool_spans: int = 48) -> Workload:
    """Long-context decode: contexts of ``n_spans`` spans drawn uniformly with
    replacement from a pool; physical block order is randomly permuted."""
    rng = np.random.default_rng(seed)
    reqs = []
    for _ in range(B):
        spans = [int(x) for x in rng.integers(0, pool_spans, size=n_spans)]
        reqs.append([("span", s, span_tokens) for s in spans])
    return build_workload(
        "long_decode", seed, dtype, Hq, Hkv, d, rope_base,
        pool_spans=pool_spans, span_tokens=span_tokens, decode_requests=reqs, rng=rng,
        notes=f"B={B} ctx={n_spans * span_tokens}: uniform spans of {span_tokens} from {pool_spans}")


def mixed_batch(seed: int = 0, dtype: str = "bf16", n_prefill: int = 16,
                chunk: int = 2048, n_decode: int = 128, min_ctx: int = 2048,
                max_ctx: int = 32768, Hq: int = 28, Hkv: int = 4, d: int = 128,
                rope_base: float = 1000000.0, span_tokens: int = 1024,
                pool_spans: int = 128, zipf_s: float = 1.1) -> Workload:
    """Mixed continuous batch: span-prefill chunks (causal within themselves
    from offset 0) and decode tokens over Zipf-drawn span contexts whose
    lengths are uniform in [min_ctx, max_ctx]; the last span is truncated."""
    rng = np.random.default_rng(seed)
    rank_to_id = rng.permutation(pool_spans)
    dec = []
    for _ in range(n_decode):
        L = int(rng.integers(min_ctx, max_ctx + 1))
        ns = -(-L // span_tokens)
        spans = _zipf_draw(rng, pool_spans, ns, zipf_s, rank_to_id)
        segs = []
        left = L
        for s in spans:
            n = min(span_tokens, left)
            segs.append(("span", s, n))
            left -= n
        dec.append(segs)
    pre = [([("own", chunk)], chunk) for _ in range(n_prefill)]
    return build_workload(
        "mixed_batch", seed, dtype, Hq, Hkv, d, rope_base,
        pool_spans=pool_spans, span_tokens=span_tokens,
        decode_requests=dec, prefill_requests=pre, rng=rng,
        notes=f"{n_prefill}x{chunk} span prefill + {n_decode} decodes, ctx U[{min_ctx},{max_ctx}]")


CONFIG_NAMES = ("tiny_decode", "rag_decode", "rag_prefill", "long_decode", "mixed_batch")


def append_case(seed: int = 0, dtype: str = "bf16", d: int = 64, Hkv: int = 2,
                seq_lens: Sequence[int] = (5, 16, 31, 0), n_new: Sequence[int] = (20, 1, 17, 3),
                pool_blocks: Optional[int] = None):
    """A cache-append case: requests holding ``seq_lens`` keys in distinct random
    physical blocks (a request owns the slots it appends into), random block
    starts, tables wide enough for ``n_new`` more keys, and the new unrotated
    keys and values.  Returns (workload, k_new, v_new, cu_new, kv_start)."""
    rng = np.random.default_rng(seed + 100)
    seq = np.asarray(seq_lens, dtype=np.int32)
    nn = np.asarray(n_new, dtype=np.int64)
    B = len(seq)
    need = int(((seq + nn + BLOCK_SIZE - 1) // BLOCK_SIZE).max()) if B else 1
    nblk = pool_blocks or B * need + 4
    perm = rng.permutation(nblk).astype(np.int32)
    bt = perm[:B * need].reshape(B, need)
    st = rng.integers(0, 4096 - BLOCK_SIZE, size=(B, need)).astype(np.int32)
    k = _normal(rng, (nblk, Hkv, BLOCK_SIZE, d), dtype)
    v = _normal(rng, (nblk, Hkv, BLOCK_SIZE, d), dtype)
    q = _normal(rng, (B, 2 * Hkv, d), dtype)
    dec = DecodeBatch(q=q, block_tables=bt, block_starts=st, seq_lens=seq,
                      q_pos=rng.integers(0, 4096, size=B).astype(np.int32))
    w = Workload("append_case", dtype, 2 * Hkv, Hkv, d, BLOCK_SIZE, 10000.0, 4096, PagedKV(k, v), decode=dec)
    cu = np.concatenate([[0], np.cumsum(nn)]).astype(np.int64)
    shape = (int(cu[-1]), Hkv, d)
    return w, _normal(rng, shape, dtype), _normal(rng, shape, dtype), cu, seq.astype(np.int64)


def config(index: int, seed: int = 0, dtype: Optional[str] = None, **kw) -> Workload:
    """The five workloads by index 0..4 (full sizes unless overridden)."""
    if index == 0:
        return tiny_decode(seed, dtype or "f32")
    if index == 1:
        return rag_decode(seed, dtype or "bf16", **kw)
    if index == 2:
        return rag_prefill(seed, dtype or "bf16", **kw)
    if index == 3:
        return long_decode(seed, dtype or "bf16", **kw)
    if index == 4:
        return mixed_batch(seed, dtype or "bf16", **kw)
    raise IndexError(index)


# ----------------------------------------------------------------------------
# Irregular cases for edge tests: arbitrary per-block start positions
# ----------------------------------------------------------------------------

def irregular_decode(seed: int, dtype: str, seq_lens: Sequence[int], Hq: int = 8,
                     Hkv: int = 2, d: int = 128, rope_base: float = 10000.0,
                     max_pos: int = 4096, pool_blocks: Optional[int] = None) -> Workload:
    """Decode with random physical blocks (repeats allowed, also within one
    request) and random, non-contiguous, possibly repeated or decreasing block
    start positions and query positions; ``seq_lens`` may hold 0 and ragged
    lengths."""
    rng = np.random.default_rng(seed)
    bs = BLOCK_SIZE
    seq = np.asarray(seq_lens, dtype=np.int32)
    B = len(seq)
    nb = np.maximum(1, -(-seq // bs))
    mb = int(nb.max()) if B else 1
    nblk = pool_blocks or max(4, int(nb.sum()) // 2 + 1)
    bt = np.full((B, mb), -1, dtype=np.int32)
    st = np.zeros((B, mb), dtype=np.int32)
    for r in range(B):
        n = -(-int(seq[r]) // bs)
        bt[r, :n] = rng.integers(0, nblk, size=n)
        st[r, :n] = rng.integers(0, max_pos - bs + 1, size=n)
    qpos = rng.integers(0, max_pos, size=B).astype(np.int32)
    k = _normal(rng, (nblk, Hkv, bs, d), dtype)
    v = _normal(rng, (nblk, Hkv, bs, d), dtype)
    q = _normal(rng, (B, Hq, d), dtype)
    dec = DecodeBatch(q=q, block_tables=bt, block_starts=st, seq_lens=seq, q_pos=qpos)
    used = set(int(x) for x in np.unique(bt) if x >= 0)
    return Workload("irregular_decode", dtype, Hq, Hkv, d, bs, float(rope_base), int(max_pos),
                    PagedKV(k, v), decode=dec, notes="random starts/blocks", unique_blocks=len(used))


def irregular_prefill(seed: int, dtype: str, kv_lens: Sequence[int], q_lens: Sequence[int],
                      Hq: int = 8, Hkv: int = 2, d: int = 128, rope_base: float = 10000.0,
                      max_pos: int = 4096, pool_blocks: Optional[int] = None) -> Workload:
    """Prefill with random physical blocks and random per-block start
    positions; query positions are random too (the causal rule is by key index,
    so positions need not be ordered)."""
    rng = np.random.default_rng(seed)
    bs = BLOCK_SIZE
    kv = np.asarray(kv_lens, dtype=np.int32)
    ql = np.asarray(q_lens, dtype=np.int32)
    assert np.all(ql <= kv)
    B = len(kv)
    nb = np.maximum(1, -(-kv // bs))
    mb = int(nb.max()) if B else 1
    nblk = pool_blocks or max(4, int(nb.sum()) // 2 + 1)
    bt = np.full((B, mb), -1, dtype=np.int32)
    st = np.zeros((B, mb), dtype=np.int32)
    for r in range(B):
        n = -(-int(kv[r]) // bs)
        bt[r, :n] = rng.integers(0, nblk, size=n)
        st[r, :n] = rng.integers(0, max_pos - bs + 1, size=n)
    cu = np.zeros(B + 1, dtype=np.int32)
    cu[1:] = np.cumsum(ql)
    qpos = rng.integers(0, max_pos, size=int(cu[-1])).astype(np.int32)
    k = _normal(rng, (nblk, Hkv, bs, d), dtype)
    v = _normal(rng, (nblk, Hkv, bs, d), dtype)
    q = _normal(rng, (int(cu[-1]), Hq, d), dtype)
    pre = PrefillBatch(q=q, cu_q_lens=cu, q_pos=qpos, kv_lens=kv, block_tables=bt, block_starts=st)
    used = set(int(x) for x in np.unique(bt) if x >= 0)
    return Workload("irregular_prefill", dtype, Hq, Hkv, d, bs, float(rope_base), int(max_pos),
                    PagedKV(k, v), prefill=pre, notes="random starts/blocks", unique_blocks=len(used))
