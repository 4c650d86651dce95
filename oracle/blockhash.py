"""Block hashing with span separators, and the prefix-cache mapping it drives
(oracle; test infrastructure only).

MiniPIC summary (gist.science 2606.13126), section 2.2: KV blocks are cached
by a hash chain over their tokens, and two special tokens placed at the start
of a block change the chain:
  * default:  h_i = H(h_{i-1}, x_i)      (the block depends on every block since
                                          the chain last restarted)
  * SSEP:     h_i = H(h_0, x_i)          (the chain restarts: the span is cached
                                          whatever precedes it)
  * PDEP:     h_i = H(h_0, x_{<=i})      (the block depends on the whole prompt
                                          before it, across restarts)
with h_0 the chain's root and x_i the tokens of block i.  Padding brings spans
to block boundaries so that the special tokens open blocks (item 1 there).

Readings of what the pages leave open (listed in the design notes):
  * H is 64-bit FNV-1a over the parent hash (8 bytes, little endian) followed
    by the tokens (4 bytes each, little endian, int32);
  * only full blocks are hashed and shared; a trailing partial block is
    private to its request;
  * the prefix cache maps a hash to one physical block; a request's block b
    sits at logical positions b * block_size .. (the position-free cache lets
    the same physical block serve other requests at other offsets);
  * a miss takes the lowest never-used block id, else evicts the released
    (unreferenced) block that was released longest ago.
"""

from __future__ import annotations

from collections import OrderedDict
from typing import List, Optional, Sequence, Tuple

import numpy as np

FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
_MASK = (1 << 64) - 1


def fnv1a64(data: bytes, h: int = FNV_OFFSET) -> int:
    """64-bit FNV-1a: for each byte, h ^= byte, then h *= prime (mod 2^64)."""
    for b in data:
        h ^= b
        h = (h * FNV_PRIME) & _MASK
    return h


def chain_hash(parent: int, tokens: Sequence[int]) -> int:
    """H(parent, tokens)."""
    data = int(parent).to_bytes(8, "little")
    for t in tokens:
        data += int(t).to_bytes(4, "little", signed=True)
    return fnv1a64(data)


def block_hashes(tokens: Sequence[int], block_size: int, ssep: int, pdep: int, h0: int) -> List[int]:
    """Hash of every full block of a prompt, by the rules above."""
    toks = [int(t) for t in tokens]
    n_full = len(toks) // block_size
    out: List[int] = []
    prev = h0
    for i in range(n_full):
        x = toks[i * block_size:(i + 1) * block_size]
        if x[0] == ssep:
            h = chain_hash(h0, x)
        elif x[0] == pdep:
            h = chain_hash(h0, toks[:(i + 1) * block_size])
        else:
            h = chain_hash(prev, x)
        out.append(h)
        prev = h
    return out


class PrefixCache:
    """Hash -> physical block map over a pool of num_blocks blocks."""

    def __init__(self, num_blocks: int):
        self.num_blocks = num_blocks
        self.next_fresh = 0
        self.by_hash = {}            # hash -> block id
        self.hash_of = {}            # block id -> hash (cached blocks)
        self.refs = [0] * num_blocks
        self.released: "OrderedDict[int, None]" = OrderedDict()  # unreferenced cached blocks, oldest first

    def _take(self) -> Optional[int]:
        if self.next_fresh < self.num_blocks:
            b = self.next_fresh
            self.next_fresh += 1
            return b
        if self.released:
            b, _ = self.released.popitem(last=False)
            h = self.hash_of.pop(b, None)
            if h is not None:
                del self.by_hash[h]
            return b
        return None

    def assign(self, hashes: Sequence[int], n_blocks: int, block_size: int
               ) -> Optional[Tuple[np.ndarray, np.ndarray, np.ndarray]]:
        """Physical block, logical start and "must be computed" flag of each of
        a request's n_blocks blocks (the first len(hashes) are full and shared
        through the cache, the rest private); None when the pool runs out (the
        cache is then unchanged)."""
        table = np.full(n_blocks, -1, dtype=np.int32)
        new = np.zeros(n_blocks, dtype=np.uint8)
        snapshot = (self.next_fresh, dict(self.by_hash), dict(self.hash_of), list(self.refs),
                    OrderedDict(self.released))
        for b in range(n_blocks):
            h = hashes[b] if b < len(hashes) else None
            if h is not None and h in self.by_hash:
                blk = self.by_hash[h]
                self.released.pop(blk, None)
            else:
                blk = self._take()
                if blk is None:
                    (self.next_fresh, self.by_hash, self.hash_of, self.refs, self.released) = snapshot
                    return None
                new[b] = 1
                if h is not None:
                    self.by_hash[h] = blk
                    self.hash_of[blk] = h
            self.refs[blk] += 1
            table[b] = blk
        starts = (np.arange(n_blocks, dtype=np.int64) * block_size).astype(np.int32)
        return table, starts, new

    def release(self, block_ids: Sequence[int]) -> None:
        """Drop one reference to each block; an unreferenced cached block stays
        findable until it is evicted, a private one returns to the free list
        (as the most recently released)."""
        for b in block_ids:
            b = int(b)
            self.refs[b] -= 1
            if self.refs[b] == 0:
                self.released[b] = None
