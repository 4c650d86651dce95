"""Paged attention over unrotated keys, float64 (oracle; test infrastructure).

Follows the MiniPIC summary (gist.science 2606.13126, section 2.1, the score
equation): for query token t at position p_t and stored key j of the same
request at logical position pi(j),

    s_j = (R_{p_t} q_t) . (R_{pi(j)} k~_j) / sqrt(d)
    o_t = sum_j softmax(s)_j v_j

The key set is every stored key of the request for a decode token, and the
keys up to the query's own index for a prefill chunk (bottom-right aligned by
index).  The oracle gathers each request's keys through its block table, forms
pi(j) = block_starts[r][j // bs] + j % bs, rotates with ``rope_rotate`` and
runs a plain softmax.  Nothing here is blocked, split or fused.
"""

from __future__ import annotations

import math
from typing import Iterable, Optional

import numpy as np

from .rope import rope_rotate


def widen(x: np.ndarray, dtype: str) -> np.ndarray:
    """Input storage -> float64.  bf16 inputs arrive as uint16 bit patterns."""
    if dtype == "bf16":
        b = np.ascontiguousarray(x, dtype=np.uint16)
        return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def key_index_map(block_table_row, block_start_row, n_keys: int, block_size: int):
    """For request-local key indices j = 0 .. n_keys-1 return
    (physical block, slot, logical position) as int64 arrays:
    block = table[j // bs], slot = j % bs, pi(j) = starts[j // bs] + j % bs."""
    j = np.arange(n_keys, dtype=np.int64)
    b = j // block_size
    slot = j % block_size
    phys = np.asarray(block_table_row, dtype=np.int64)[b]
    pos = np.asarray(block_start_row, dtype=np.int64)[b] + slot
    return phys, slot, pos


def attend(q_rot: np.ndarray, k_rot: np.ndarray, v: np.ndarray, scale: float,
           allowed: Optional[np.ndarray] = None):
    """Plain softmax attention in float64.

    q_rot [m, d], k_rot [n, d], v [n, d]; ``allowed`` [m, n] masks keys.
    Returns (out [m, d], lse [m]); a row with no allowed key gives zeros and
    lse = -inf."""
    m = q_rot.shape[0]
    n = k_rot.shape[0]
    dv = v.shape[1]
    out = np.zeros((m, dv), dtype=np.float64)
    lse = np.full(m, -np.inf, dtype=np.float64)
    if n == 0 or m == 0:
        return out, lse
    s = (q_rot @ k_rot.T) * scale
    if allowed is not None:
        s = np.where(allowed, s, -np.inf)
    mx = np.max(s, axis=1)
    ok = np.isfinite(mx)
    if not np.any(ok):
        return out, lse
    e = np.zeros_like(s)
    e[ok] = np.exp(s[ok] - mx[ok, None])
    l = e.sum(axis=1)
    out[ok] = (e[ok] @ v) / l[ok, None]
    lse[ok] = mx[ok] + np.log(l[ok])
    return out, lse


def _scale(w, scale):
    return (1.0 / math.sqrt(w.d)) if not scale else float(scale)


def _gathered(w, table_row, start_row, n_keys, g):
    """Gather request keys/values of kv head g; returns (k~ [n,d], v [n,d], pi [n])."""
    phys, slot, pos = key_index_map(table_row, start_row, n_keys, w.block_size)
    k = widen(w.kv.k_pool[phys, g, slot], w.dtype)
    v = widen(w.kv.v_pool[phys, g, slot], w.dtype)
    return k, v, pos


def decode(w, requests: Optional[Iterable[int]] = None, scale: float = 0.0):
    """Decode outputs for the requested requests (all by default).

    Returns (out [B, Hq, d], lse [B, Hq]); rows of requests not asked for stay
    NaN.  Work is done per (request, kv head): the keys are gathered and rotated
    once and the G query heads of that kv head are scored against them."""
    dec = w.decode
    B = dec.batch
    G = w.Hq // w.Hkv
    out = np.full((B, w.Hq, w.d), np.nan)
    lse = np.full((B, w.Hq), np.nan)
    sc = _scale(w, scale)
    for r in (range(B) if requests is None else requests):
        n = int(dec.seq_lens[r])
        qr = rope_rotate(widen(dec.q[r], w.dtype), [int(dec.q_pos[r])] * w.Hq, w.rope_base)
        phys, slot, pos = key_index_map(dec.block_tables[r], dec.block_starts[r], n, w.block_size)
        # all kv heads of the request at once: [Hkv, n, d], rotated at pos
        k = np.swapaxes(widen(w.kv.k_pool[phys, :, slot], w.dtype), 0, 1)
        v = np.swapaxes(widen(w.kv.v_pool[phys, :, slot], w.dtype), 0, 1)
        kr = rope_rotate(k, pos, w.rope_base)
        for g in range(w.Hkv):
            o, l = attend(qr[g * G:(g + 1) * G], kr[g], v[g], sc)
            out[r, g * G:(g + 1) * G] = o
            lse[r, g * G:(g + 1) * G] = l
    return out, lse


def prefill_request(w, r: int, scale: float = 0.0, heads: Optional[Iterable[int]] = None):
    """Prefill outputs of request r: (out [q_len, Hq, d], lse [q_len, Hq]).

    Query i of the chunk (i = 0 .. q_len-1) attends keys j <= kv_len - q_len + i."""
    pre = w.prefill
    G = w.Hq // w.Hkv
    q0, q1 = int(pre.cu_q_lens[r]), int(pre.cu_q_lens[r + 1])
    ql = q1 - q0
    kv = int(pre.kv_lens[r])
    sc = _scale(w, scale)
    out = np.full((ql, w.Hq, w.d), np.nan)
    lse = np.full((ql, w.Hq), np.nan)
    if ql == 0:
        return out, lse
    i = np.arange(ql)[:, None]
    j = np.arange(kv)[None, :]
    allowed = j <= (kv - ql + i)
    qpos = pre.q_pos[q0:q1]
    hs = range(w.Hq) if heads is None else list(heads)
    for g in sorted(set(h // G for h in hs)):
        k, v, pos = _gathered(w, pre.block_tables[r], pre.block_starts[r], kv, g)
        kr = rope_rotate(k, pos, w.rope_base)
        for h in hs:
            if h // G != g:
                continue
            qr = rope_rotate(widen(pre.q[q0:q1, h], w.dtype), qpos, w.rope_base)
            o, l = attend(qr, kr, v, sc, allowed)
            out[:, h] = o
            lse[:, h] = l
    return out, lse


def prefill(w, requests: Optional[Iterable[int]] = None, scale: float = 0.0):
    """Prefill outputs for all (or the given) requests, packed like q:
    (out [total_q, Hq, d], lse [total_q, Hq]); rows not computed stay NaN."""
    pre = w.prefill
    tq = int(pre.cu_q_lens[-1])
    out = np.full((tq, w.Hq, w.d), np.nan)
    lse = np.full((tq, w.Hq), np.nan)
    for r in (range(pre.batch) if requests is None else requests):
        q0, q1 = int(pre.cu_q_lens[r]), int(pre.cu_q_lens[r + 1])
        o, l = prefill_request(w, r, scale)
        out[q0:q1] = o
        lse[q0:q1] = l
    return out, lse
