"""The float64 oracle over many requests at once, on every host core.

Test infrastructure for the full-size parity tests: one spawned worker process
per core (BLAS held to one thread in each), all reading the workload's KV pool
from shared memory, each scoring whole requests with the oracle.  Results come
back as the same arrays ``oracle.decode`` / ``oracle.prefill`` return (rows of
requests not asked for stay NaN).
"""

from __future__ import annotations

import multiprocessing as mproc
import os
from multiprocessing import shared_memory

import numpy as np

_W = None
_SHM = []


_BLAS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")


def _init(spec):
    global _W
    import workloads as W
    pools = []
    for name, shape, dtype in spec["pools"]:
        shm = shared_memory.SharedMemory(name=name)
        _SHM.append(shm)
        pools.append(np.ndarray(shape, dtype=dtype, buffer=shm.buf))
    _W = W.Workload(spec["name"], spec["dtype"], spec["Hq"], spec["Hkv"], spec["d"], spec["block_size"],
                    spec["rope_base"], spec["max_pos"], W.PagedKV(pools[0], pools[1]),
                    decode=W.DecodeBatch(**spec["decode"]) if spec["decode"] else None,
                    prefill=W.PrefillBatch(**spec["prefill"]) if spec["prefill"] else None)


def _decode_one(r):
    import oracle
    out, lse = oracle.decode(_W, requests=[r])
    return r, out[r], lse[r]


def _prefill_one(r):
    import oracle
    out, lse = oracle.prefill_request(_W, r)
    return r, out, lse


class OraclePool:
    def __init__(self, w, n_workers=None):
        self.w = w
        self.shm = []
        pools = []
        for a in (w.kv.k_pool, w.kv.v_pool):
            shm = shared_memory.SharedMemory(create=True, size=max(1, a.nbytes))
            np.ndarray(a.shape, dtype=a.dtype, buffer=shm.buf)[...] = a
            self.shm.append(shm)
            pools.append((shm.name, a.shape, a.dtype.str))
        d, p = w.decode, w.prefill
        spec = dict(name=w.name, dtype=w.dtype, Hq=w.Hq, Hkv=w.Hkv, d=w.d, block_size=w.block_size,
                    rope_base=w.rope_base, max_pos=w.max_pos, pools=pools,
                    decode=None if d is None else dict(q=d.q, block_tables=d.block_tables,
                                                       block_starts=d.block_starts, seq_lens=d.seq_lens,
                                                       q_pos=d.q_pos),
                    prefill=None if p is None else dict(q=p.q, cu_q_lens=p.cu_q_lens, q_pos=p.q_pos,
                                                        kv_lens=p.kv_lens, block_tables=p.block_tables,
                                                        block_starts=p.block_starts))
        self.n = int(n_workers or os.cpu_count() or 1)
        saved = {k: os.environ.get(k) for k in _BLAS}
        os.environ.update({k: "1" for k in _BLAS})  # inherited by the workers, whose BLAS then runs one thread
        try:
            self.pool = mproc.get_context("spawn").Pool(self.n, initializer=_init, initargs=(spec,))
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def decode(self, requests):
        d = self.w.decode
        out = np.full((d.batch, self.w.Hq, self.w.d), np.nan)
        lse = np.full((d.batch, self.w.Hq), np.nan)
        for r, o, l in self.pool.imap_unordered(_decode_one, list(requests)):
            out[r], lse[r] = o, l
        return out, lse

    def prefill(self, requests):
        p = self.w.prefill
        tq = int(p.cu_q_lens[-1])
        out = np.full((tq, self.w.Hq, self.w.d), np.nan)
        lse = np.full((tq, self.w.Hq), np.nan)
        for r, o, l in self.pool.imap_unordered(_prefill_one, list(requests)):
            q0, q1 = int(p.cu_q_lens[r]), int(p.cu_q_lens[r + 1])
            out[q0:q1], lse[q0:q1] = o, l
        return out, lse

    def close(self):
        self.pool.close()
        self.pool.join()
        for shm in self.shm:
            shm.close()
            shm.unlink()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
