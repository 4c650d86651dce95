"""Block offload on the GPU (through the C ABI): swap-out fills pinned host
buffers with exactly the listed blocks; swap-in writes them back bit for bit,
to the same or to other physical ids; decode over blocks relocated this way
with only the tables remapped matches the oracle (no position fix-up)."""

import numpy as np
import pytest

import oracle
from oracle import cache
import workloads as W
from gpu_util import compare, compare_lse

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


def to_dev(torch, dev, a, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


def bits(torch, t, dtype):
    t = t.cpu() if t.is_cuda else t
    return t.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else t.numpy()


def i32(torch, dev, a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 64)])
def test_swap_out_and_back_in_bit_for_bit(env, dtype, d):
    torch, mp, dev = env
    rng = np.random.default_rng(d)
    nblk, Hkv = 40, 4
    k = W._normal(rng, (nblk, Hkv, 16, d), dtype)
    v = W._normal(rng, (nblk, Hkv, 16, d), dtype)
    kp, vp = to_dev(torch, dev, k, dtype), to_dev(torch, dev, v, dtype)
    ids = rng.choice(nblk, size=13, replace=False)
    hk, hv = mp.kv_swap_out(kp, vp, i32(torch, dev, ids))
    torch.cuda.synchronize()
    ek, ev = cache.swap_out(k, v, ids)
    assert np.array_equal(bits(torch, hk, dtype), ek) and np.array_equal(bits(torch, hv, dtype), ev)
    # clobber, then bring them back to a permutation of other ids
    kp.zero_()
    vp.zero_()
    dest = rng.permutation(np.setdiff1d(np.arange(nblk), ids))[:len(ids)]
    mp.kv_swap_in(hk, hv, i32(torch, dev, dest), kp, vp)
    torch.cuda.synchronize()
    rk, rv = cache.swap_in(np.zeros_like(k), np.zeros_like(v), ek, ev, dest)
    assert np.array_equal(bits(torch, kp, dtype), rk) and np.array_equal(bits(torch, vp, dtype), rv)
    assert mp.device_error() == 0


def test_bad_ids_are_flagged_and_skipped(env):
    torch, mp, dev = env
    rng = np.random.default_rng(1)
    k = W._normal(rng, (8, 2, 16, 64), "bf16")
    kp, vp = to_dev(torch, dev, k, "bf16"), to_dev(torch, dev, k, "bf16")
    mp.device_error(clear=True)
    hk, hv = mp.kv_swap_out(kp, vp, i32(torch, dev, [3, 99, 5]))
    torch.cuda.synchronize()
    assert mp.device_error(clear=True) & 1
    got = bits(torch, hk, "bf16")
    assert np.array_equal(got[0], k[3]) and np.array_equal(got[2], k[5])


def test_relocated_blocks_decode_like_the_oracle(env):
    """Swap a request's blocks out, bring them back to fresh physical ids, remap
    the tables (starts untouched) and decode on the GPU: as the oracle decodes
    the original cache."""
    torch, mp, dev = env
    w = W.rag_decode(6, "bf16", B=4, Hq=8, Hkv=2, d=128, system_tokens=32, n_spans=3, span_tokens=64,
                     pool_spans=6, tail_tokens=32)
    d = w.decode
    ref, ref_lse = oracle.decode(w)
    n0 = -(-int(d.seq_lens[0]) // 16)
    old = np.unique(d.block_tables[0, :n0])
    nb = w.kv.num_blocks
    new = np.arange(nb, nb + len(old))
    grow = lambda a: np.concatenate([a, np.zeros((len(old),) + a.shape[1:], dtype=a.dtype)])
    kp, vp = to_dev(torch, dev, grow(w.kv.k_pool), "bf16"), to_dev(torch, dev, grow(w.kv.v_pool), "bf16")
    hk, hv = mp.kv_swap_out(kp, vp, i32(torch, dev, old))
    torch.cuda.synchronize()
    kp[torch.from_numpy(old).to(dev)] = 0  # the device copies are gone
    vp[torch.from_numpy(old).to(dev)] = 0
    mp.kv_swap_in(hk, hv, i32(torch, dev, new), kp, vp)
    tables = cache.remap_tables(d.block_tables, old, new)
    rope = mp.rope_table(w.max_pos, w.d, w.rope_base, device=dev)
    lse = torch.full((d.batch, w.Hq), float("nan"), device=dev)
    out, _ = mp.attn_decode(to_dev(torch, dev, d.q, "bf16"), kp, vp, i32(torch, dev, tables),
                            i32(torch, dev, d.block_starts), i32(torch, dev, d.seq_lens),
                            i32(torch, dev, d.q_pos), rope, lse=lse)
    torch.cuda.synchronize()
    compare(out.float().cpu().numpy(), ref, "bf16", "decode after relocation")
    compare_lse(lse.cpu().numpy(), ref_lse, "bf16", "decode after relocation")
    assert mp.device_error() == 0
