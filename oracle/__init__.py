"""CPU float64 oracle for position-free paged attention (MiniPIC).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test-suite, the package
smoke check and the benchmark's CPU-baseline leg may import or run anything in
this package.  The CUDA library never calls it and shares no code with it.

What it computes is the plain definition from the MiniPIC summary page
(gist.science paper 2606.13126, section 2.1, the score equation): keys are
stored unrotated, and the score of query token t against stored key j is

    score(t, j) = (R_t q_t)^T (R_{pi(j)} k~_j) / sqrt(d)

with pi(j) the logical position of key j inside the current request, followed
by an ordinary softmax-weighted sum of the (unrotated) values.  The same page
states that this is algebraically the same as re-rotating a cache hit to its
new offset (section 2.1, "Implementazione"); the oracle is written as that plain
definition, in float64, with rotary angles formed in extended precision.

Readings of points the pages leave open (each is listed in the design notes):
  * rotary pairing: half rotation, element i pairs with element i + d/2;
  * frequencies: theta_i = base^(-2 i / d), i < d/2, no frequency scaling;
  * pi(j) = block_starts[r][j // bs] + j % bs;
  * GQA: query head h reads kv head h // (Hq / Hkv);
  * values are not rotated; scale defaults to 1/sqrt(d);
  * prefill causality is by key index, bottom-right aligned: query i of a
    q_len chunk sees keys j <= kv_len - q_len + i;
  * an empty key set gives output 0 and log-sum-exp -inf.

``oracle.blockhash`` holds the host-side step that feeds the attention its
tables: the block-hash chain with span separators (SSEP restarts the chain,
PDEP ties a block to the whole prompt before it; MiniPIC summary section 2.2)
and the prefix-cache mapping from hashes to physical blocks.
"""

from .rope import inv_freq, rope_angles, rope_cos_sin, rope_table, rope_rotate
from .attention import (
    widen,
    key_index_map,
    attend,
    decode,
    prefill_request,
    prefill,
)

__all__ = [
    "inv_freq",
    "rope_angles",
    "rope_cos_sin",
    "rope_table",
    "rope_rotate",
    "widen",
    "key_index_map",
    "attend",
    "decode",
    "prefill_request",
    "prefill",
]
