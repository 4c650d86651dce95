"""Helpers for the GPU tests: upload seeded workloads and compare with the oracle."""

import numpy as np

TOL = {"f32": dict(max_abs=1e-4, mean_abs=1e-4, lse=1e-4),
       "bf16": dict(max_abs=1e-2, mean_abs=1e-3, lse=2e-2)}


def to_dev(a, dtype, torch, dev):
    """Workload storage (float32 or bf16 bits) -> CUDA tensor of the path's dtype."""
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


def i32(a, torch, dev):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def upload_decode(w, torch, dev):
    d = w.decode
    return dict(q=to_dev(d.q, w.dtype, torch, dev), k_pool=to_dev(w.kv.k_pool, w.dtype, torch, dev),
                v_pool=to_dev(w.kv.v_pool, w.dtype, torch, dev),
                block_tables=i32(d.block_tables, torch, dev), block_starts=i32(d.block_starts, torch, dev),
                seq_lens=i32(d.seq_lens, torch, dev), q_pos=i32(d.q_pos, torch, dev))


def upload_prefill(w, torch, dev):
    p = w.prefill
    return dict(q=to_dev(p.q, w.dtype, torch, dev), k_pool=to_dev(w.kv.k_pool, w.dtype, torch, dev),
                v_pool=to_dev(w.kv.v_pool, w.dtype, torch, dev), cu_q_lens=i32(p.cu_q_lens, torch, dev),
                q_pos=i32(p.q_pos, torch, dev), kv_lens=i32(p.kv_lens, torch, dev),
                block_tables=i32(p.block_tables, torch, dev), block_starts=i32(p.block_starts, torch, dev))


def compare(got, ref, dtype, what=""):
    """Element-wise comparison against the oracle on the rows it computed."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    mask = ~np.isnan(ref)
    assert mask.any(), "no reference rows"
    diff = np.abs(got[mask] - ref[mask])
    tol = TOL[dtype]
    mx, mean = float(diff.max()), float(diff.mean())
    assert np.all(np.isfinite(got[mask])), f"{what}: non-finite output"
    assert mx <= tol["max_abs"], f"{what}: max abs err {mx:.3g} > {tol['max_abs']}"
    assert mean <= tol["mean_abs"], f"{what}: mean abs err {mean:.3g} > {tol['mean_abs']}"
    return mx, mean


def compare_lse(got, ref, dtype, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    mask = ~np.isnan(ref)
    fin = np.isfinite(ref[mask])
    assert np.array_equal(np.isfinite(got[mask]), fin), f"{what}: -inf pattern differs"
    if fin.any():
        d = np.abs(got[mask][fin] - ref[mask][fin]).max()
        assert d <= TOL[dtype]["lse"], f"{what}: lse err {d:.3g}"
