"""Inputs whose attention output spells out which keys were read.

Used by the exact-indexing tests.  With every visible key weighted equally
(a zero query, or keys that all score the same), the output of a query row is
the mean of the value rows it gathered.  If each value row is a small integer
code of (physical block, slot, kv head), the mean times the number of keys is
a vector of integer counts, so the set of (block, slot) pairs a kernel visited
can be read back exactly and compared with the oracle's.

Value row of (physical block b, kv head g, slot s), head dim d:
    e_s                     (slot one-hot, dims 0..15)
  + e_{16 + b}              (block one-hot, dims 16..d-2; needs num_blocks <= d - 17)
  + (g + 1) e_{d-1}         (kv head tag)
so, for a row that attends n keys, n * out[:16] counts the keys per slot,
n * out[16:d-1] counts the keys per physical block, and out[d-1] = g + 1.
"""

from __future__ import annotations

import numpy as np

import oracle
import workloads as W


def coded_values(num_blocks: int, Hkv: int, bs: int, d: int, dtype: str) -> np.ndarray:
    """Value pool [num_blocks, Hkv, bs, d] holding the codes above, in the
    workload's storage (float32, or bf16 bit patterns; every code is exact)."""
    if num_blocks > d - 17 or bs > 16:
        raise ValueError("codes need num_blocks <= d - 17 and block_size <= 16")
    v = np.zeros((num_blocks, Hkv, bs, d), dtype=np.float32)
    for b in range(num_blocks):
        for g in range(Hkv):
            for s in range(bs):
                v[b, g, s, s] = 1.0
                v[b, g, s, 16 + b] = 1.0
                v[b, g, s, d - 1] = float(g + 1)
    return W.to_bf16_bits(v) if dtype == "bf16" else v


def counts(out_row: np.ndarray, n_keys: int):
    """(integer counts, largest distance of n*out from an integer) of one row."""
    x = np.asarray(out_row, dtype=np.float64)[:-1] * float(n_keys)
    r = np.rint(x)
    return r.astype(np.int64), float(np.abs(x - r).max()) if x.size else 0.0


def counts_from_indices(phys: np.ndarray, slot: np.ndarray, d: int) -> np.ndarray:
    """The counts the codes give for a gathered key set, from its indices."""
    c = np.zeros(d - 1, dtype=np.int64)
    np.add.at(c, np.asarray(slot, dtype=np.int64), 1)
    np.add.at(c, 16 + np.asarray(phys, dtype=np.int64), 1)
    return c


def phase_margin(d: int, base: float, n_pairs: int, max_shift: int) -> float:
    """max over shifts 1 <= delta <= max_shift of the mean of cos(delta theta_i)
    over the first n_pairs rotary frequencies: the largest score fraction a
    key keeps when a kernel rotates it delta positions away from where it was
    aligned (see ``align_keys``)."""
    i = np.arange(n_pairs, dtype=np.float64)
    theta = np.power(float(base), -2.0 * i / d)
    delta = np.arange(1, max_shift + 1, dtype=np.float64)[:, None]
    return float(np.cos(delta * theta[None, :]).mean(axis=1).max())


def unit_direction(rng: np.random.Generator, d: int, n_pairs: int) -> np.ndarray:
    """Unit vector with equal energy in each of the first n_pairs rotary pairs
    (element i pairs with i + d/2) and nothing elsewhere."""
    u = np.zeros(d, dtype=np.float64)
    ang = rng.uniform(0.0, 2.0 * np.pi, size=n_pairs)
    u[:n_pairs] = np.cos(ang)
    u[d // 2:d // 2 + n_pairs] = np.sin(ang)
    return u / np.sqrt(n_pairs)


def zero_query_decode(seed: int, dtype: str, Hq: int, Hkv: int, d: int, seq_lens) -> W.Workload:
    """Decode batch with random block ids (repeats allowed) and random starts,
    q = 0 and coded value rows."""
    w = W.irregular_decode(seed, dtype, seq_lens=seq_lens, Hq=Hq, Hkv=Hkv, d=d, max_pos=70000,
                           pool_blocks=d - 17)
    w.decode.q[:] = 0
    w.kv.v_pool = coded_values(w.kv.num_blocks, Hkv, w.block_size, d, dtype)
    return w


def zero_query_prefill(seed: int, Hq: int, Hkv: int, d: int, kv_lens, q_lens) -> W.Workload:
    """Prefill batch (bf16) with random block ids and starts, q = 0 and coded
    value rows."""
    w = W.irregular_prefill(seed, "bf16", kv_lens=kv_lens, q_lens=q_lens, Hq=Hq, Hkv=Hkv, d=d, max_pos=60000,
                            pool_blocks=d - 17)
    w.prefill.q[:] = 0
    w.kv.v_pool = coded_values(w.kv.num_blocks, Hkv, w.block_size, d, "bf16")
    return w


# phase-aligned fp32 decode: sizes and the common score M
ALIGNED = dict(d=128, Hq=8, Hkv=2, max_pos=4096, n_pairs=16, M=300.0, seq=(1, 16, 17, 90, 250, 700))


def aligned_decode(seed: int = 70, index_map=None) -> W.Workload:
    """fp32 decode in which every stored key k~_j is the direction u of its
    (request, kv head) rotated back by pi(j), and the query is u rotated back by
    its position, scaled so that a correct rotation gives every key the score
    M.  Every block is used once in the batch (a stored key is aligned for one
    position only).  ``index_map`` (default: the oracle's) gives the positions
    the keys are aligned for."""
    c = ALIGNED
    d, Hq, Hkv, seq = c["d"], c["Hq"], c["Hkv"], list(c["seq"])
    w = W.irregular_decode(seed, "f32", seq_lens=seq, Hq=Hq, Hkv=Hkv, d=d, max_pos=c["max_pos"],
                           pool_blocks=d - 17)
    dec = w.decode
    rng = np.random.default_rng(seed + 1)
    perm = rng.permutation(w.kv.num_blocks)
    k = 0
    for r in range(dec.batch):
        nb = -(-seq[r] // 16)
        dec.block_tables[r, :nb] = perm[k:k + nb]
        k += nb
    G = Hq // Hkv
    amp = np.sqrt(c["M"] * np.sqrt(d))  # scale 1/sqrt(d): score = amp^2 / sqrt(d) = M
    kpool = w.kv.k_pool.astype(np.float64)
    imap = index_map or oracle.key_index_map
    for r in range(dec.batch):
        phys, slot, pos = imap(dec.block_tables[r], dec.block_starts[r], seq[r], 16)
        for g in range(Hkv):
            u = unit_direction(rng, d, c["n_pairs"]) * amp
            q = oracle.rope_rotate(u[None, :], [-int(dec.q_pos[r])], w.rope_base)[0]
            dec.q[r, g * G:(g + 1) * G] = q.astype(np.float32)
            kpool[phys, g, slot] = oracle.rope_rotate(np.repeat(u[None, :], len(pos), 0), -pos, w.rope_base)
    w.kv.k_pool = kpool.astype(np.float32)
    w.kv.v_pool = coded_values(w.kv.num_blocks, Hkv, 16, d, "f32")
    return w
