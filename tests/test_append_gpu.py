"""Cache append on the GPU (through the C ABI) against the oracle: the pools
after the call equal oracle.cache.append bit for bit; bad table entries are
flagged and skipped; keys appended on the GPU are read back correctly by the
prefill kernel."""

import numpy as np
import pytest

import oracle
from oracle import cache
import workloads as W
from gpu_util import compare, upload_prefill

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


def dev_arr(torch, dev, a, dtype):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev)


def host_bits(torch, t, dtype):
    """Device pool -> host array in the workload's storage (bf16 as uint16 bits)."""
    if dtype == "bf16":
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def i32(torch, dev, a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


def run_append(env, w, k_new, v_new, cu, kv_start, tables=None):
    torch, mp, dev = env
    tables = w.decode.block_tables if tables is None else tables
    kp, vp = dev_arr(torch, dev, w.kv.k_pool, w.dtype), dev_arr(torch, dev, w.kv.v_pool, w.dtype)
    mp.kv_append(dev_arr(torch, dev, k_new, w.dtype), dev_arr(torch, dev, v_new, w.dtype), i32(torch, dev, cu),
                 i32(torch, dev, kv_start), i32(torch, dev, tables), kp, vp)
    torch.cuda.synchronize()
    return host_bits(torch, kp, w.dtype), host_bits(torch, vp, w.dtype)


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("bf16", 64), ("f32", 128), ("f32", 64)])
def test_append_equals_oracle_bit_for_bit(env, dtype, d):
    w, k_new, v_new, cu, kv_start = W.append_case(7 + d, dtype, d=d, Hkv=4,
                                                  seq_lens=(5, 16, 31, 0, 47), n_new=(20, 1, 17, 3, 0))
    k, v = run_append(env, w, k_new, v_new, cu, kv_start)
    kr, vr = cache.append(w.kv.k_pool, w.kv.v_pool, k_new, v_new, cu, kv_start, w.decode.block_tables)
    assert np.array_equal(k, kr) and np.array_equal(v, vr)
    assert env[1].device_error() == 0


def test_bad_table_entries_are_flagged_and_skipped(env):
    torch, mp, dev = env
    w, k_new, v_new, cu, kv_start = W.append_case(3, "bf16", d=128)
    mp.device_error(clear=True)
    tables = w.decode.block_tables.copy()
    bad_r, bad_j = 0, int(kv_start[0]) + 12  # request 0's 13th new key -> block id out of range
    tables[bad_r, bad_j // 16] = 10 ** 6
    k, v = run_append(env, w, k_new, v_new, cu, kv_start, tables)
    assert mp.device_error(clear=True) & 1
    # every key that maps to a valid block is written as the oracle writes it
    keep = np.ones(int(cu[-1]), dtype=bool)
    for i in range(int(cu[1] - cu[0])):
        if (int(kv_start[0]) + i) // 16 == bad_j // 16:
            keep[int(cu[0]) + i] = False
    # expected: the oracle's append with the keys of the bad block left out
    kr, vr = w.kv.k_pool.copy(), w.kv.v_pool.copy()
    for r in range(len(cu) - 1):
        for i in range(int(cu[r + 1] - cu[r])):
            t, j = int(cu[r]) + i, int(kv_start[r]) + i
            if not keep[t]:
                continue
            kr[tables[r][j // 16], :, j % 16] = k_new[t]
            vr[tables[r][j // 16], :, j % 16] = v_new[t]
    assert np.array_equal(k, kr) and np.array_equal(v, vr)
    # a key index beyond the table is flagged too
    too_far = kv_start.copy()
    too_far[1] = w.decode.block_tables.shape[1] * 16
    run_append(env, w, k_new, v_new, cu, too_far)
    assert mp.device_error(clear=True) & 4


def test_prefill_reads_keys_appended_on_the_gpu(env):
    """Clear the chunks' own keys, append them back with the GPU kernel, and
    run the prefill over the result: same pools, output as the oracle's."""
    torch, mp, dev = env
    w = W.rag_prefill(4, B=3, n_spans=2, span_tokens=256, pool_spans=5, q_len=200)
    p = w.prefill
    q_lens = np.diff(p.cu_q_lens).astype(np.int64)
    kv_start = p.kv_lens.astype(np.int64) - q_lens
    cu = np.concatenate([[0], np.cumsum(q_lens)])
    k_new = np.concatenate([cache.gather(w.kv.k_pool, p.block_tables[r], int(kv_start[r]), int(q_lens[r]))
                            for r in range(p.batch)])
    v_new = np.concatenate([cache.gather(w.kv.v_pool, p.block_tables[r], int(kv_start[r]), int(q_lens[r]))
                            for r in range(p.batch)])
    t = upload_prefill(w, torch, dev)
    kp, vp = t["k_pool"], t["v_pool"]
    for r in range(p.batch):  # clear the chunk slots on the device
        for j in range(int(kv_start[r]), int(p.kv_lens[r])):
            kp[int(p.block_tables[r][j // 16]), :, j % 16] = 0
            vp[int(p.block_tables[r][j // 16]), :, j % 16] = 0
    mp.kv_append(dev_arr(torch, dev, k_new, "bf16"), dev_arr(torch, dev, v_new, "bf16"), i32(torch, dev, cu),
                 i32(torch, dev, kv_start), t["block_tables"], kp, vp)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(torch, kp, "bf16"), w.kv.k_pool)
    assert np.array_equal(host_bits(torch, vp, "bf16"), w.kv.v_pool)
    rope = mp.rope_table(w.max_pos, w.d, w.rope_base, device=dev)
    out, _ = mp.attn_prefill(t["q"], t["cu_q_lens"], t["q_pos"], kp, vp, t["block_tables"], t["block_starts"],
                             t["kv_lens"], rope, max_q_len=int(q_lens.max()))
    torch.cuda.synchronize()
    ref, _ = oracle.prefill(w)
    compare(out.float().cpu().numpy(), ref, "bf16", "prefill after append")


def test_full_size_chunk_append(env):
    """The RAG prefill's 8 x 512-token chunks (8 kv heads, d 128) appended in one
    call: bit-exact against the oracle."""
    w = W.rag_prefill(0)
    p = w.prefill
    q_lens = np.diff(p.cu_q_lens).astype(np.int64)
    kv_start = p.kv_lens.astype(np.int64) - q_lens
    cu = np.concatenate([[0], np.cumsum(q_lens)])
    rng = np.random.default_rng(11)
    shape = (int(cu[-1]), w.Hkv, w.d)
    k_new = W.to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
    v_new = W.to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))
    w.decode = W.DecodeBatch(q=None, block_tables=p.block_tables, block_starts=p.block_starts,
                             seq_lens=p.kv_lens, q_pos=None)
    k, v = run_append(env, w, k_new, v_new, cu, kv_start)
    kr, vr = cache.append(w.kv.k_pool, w.kv.v_pool, k_new, v_new, cu, kv_start, p.block_tables)
    assert np.array_equal(k, kr) and np.array_equal(v, vr)
    assert env[1].device_error() == 0
