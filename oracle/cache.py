"""Appending new keys and values to the paged cache (oracle; test infrastructure).

Follows the MiniPIC summary (gist.science 2606.13126, section 2.1): the cache
holds unrotated key vectors k~_j, so a new token's key is stored exactly as the
model produced it, with no rotation at any position; its value likewise.  The
slot a key lands in is the one the attention gather reads it from: request r's
key index j lives in block block_tables[r][j // bs], slot j % bs.

Here token i of request r (rows cu_new[r] .. cu_new[r+1]-1 of the new keys) is
the request's key index j = kv_start[r] + i.  Plain loops; the pools are copied,
never modified in place.
"""

from __future__ import annotations

import numpy as np


def append(k_pool, v_pool, k_new, v_new, cu_new, kv_start, block_tables, block_size: int = 16):
    """Return (k_pool', v_pool') with every new token written to its slot.

    k_pool, v_pool: [num_blocks][Hkv][bs][d] (any dtype, bit patterns are copied);
    k_new, v_new: [total_new][Hkv][d]; cu_new: [B+1]; kv_start: [B];
    block_tables: [B][max_blocks].  Raises on an index the tables cannot hold."""
    k_out = np.array(k_pool, copy=True)
    v_out = np.array(v_pool, copy=True)
    cu_new = np.asarray(cu_new, dtype=np.int64)
    for r in range(len(cu_new) - 1):
        for i in range(int(cu_new[r + 1] - cu_new[r])):
            t = int(cu_new[r]) + i
            j = int(kv_start[r]) + i
            phys = int(block_tables[r][j // block_size])
            slot = j % block_size
            k_out[phys, :, slot, :] = k_new[t]
            v_out[phys, :, slot, :] = v_new[t]
    return k_out, v_out


def gather(pool, block_table_row, first: int, count: int, block_size: int = 16):
    """Rows [count][Hkv][d] of key indices first .. first+count-1 of one request,
    read back through its block table (the attention kernels' gather)."""
    out = []
    for j in range(first, first + count):
        out.append(pool[int(block_table_row[j // block_size]), :, j % block_size, :])
    if not out:
        return np.zeros((0,) + pool.shape[1:2] + pool.shape[3:], dtype=pool.dtype)
    return np.stack(out)


# ---------------------------------------------------------------- host offload
# MiniPIC summary (gist.science 2606.13126), section 3, item 5: unrotated blocks
# move between GPU and host with no position to track or adjust.  A block's
# logical positions live in the requests' block_starts, not in its contents or
# its physical id, so offload is a plain copy and a block may come back to any
# free physical id as long as the tables are remapped.

def swap_out(k_pool, v_pool, block_ids):
    """Host copies [n][Hkv][bs][d] of the listed blocks (K and V)."""
    ids = np.asarray(block_ids, dtype=np.int64)
    return np.array(k_pool[ids], copy=True), np.array(v_pool[ids], copy=True)


def swap_in(k_pool, v_pool, k_host, v_host, block_ids):
    """Pools with host block i written to physical block block_ids[i]."""
    k_out = np.array(k_pool, copy=True)
    v_out = np.array(v_pool, copy=True)
    for i, b in enumerate(np.asarray(block_ids, dtype=np.int64)):
        k_out[b] = k_host[i]
        v_out[b] = v_host[i]
    return k_out, v_out


def remap_tables(block_tables, old_ids, new_ids):
    """Tables with every entry old_ids[i] replaced by new_ids[i] (starts unchanged)."""
    m = {int(o): int(n) for o, n in zip(old_ids, new_ids)}
    out = np.array(block_tables, copy=True)
    for idx, b in np.ndenumerate(out):
        if int(b) in m:
            out[idx] = m[int(b)]
    return out
