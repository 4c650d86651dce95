"""The parallel oracle helper of the full-size GPU tests returns what the
oracle returns, for decode and prefill requests (CPU only)."""

import numpy as np

import oracle
import workloads as W
from oracle_pool import OraclePool


def test_pool_equals_the_oracle():
    w = W.mixed_batch(3, n_prefill=3, chunk=40, n_decode=5, min_ctx=1, max_ctx=900, Hq=8, Hkv=2, d=64)
    with OraclePool(w, n_workers=2) as op:
        d_out, d_lse = op.decode([0, 2, 4])
        p_out, p_lse = op.prefill([1, 2])
    ro, rl = oracle.decode(w, requests=[0, 2, 4])
    assert np.array_equal(d_out, ro, equal_nan=True) and np.array_equal(d_lse, rl, equal_nan=True)
    ro, rl = oracle.prefill(w, requests=[1, 2])
    assert np.array_equal(p_out, ro, equal_nan=True) and np.array_equal(p_lse, rl, equal_nan=True)
