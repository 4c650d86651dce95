"""Write worked_examples.json: tiny cases whose answers are closed forms.

Source: the score equation of the MiniPIC summary (gist.science 2606.13126,
section 2.1), score(t, j) = (R_t q_t)^T (R_{pi(j)} k~_j) / sqrt(d), followed by a
softmax over the request's keys.  With head_dim d = 2 there is a single
rotary pair with theta_0 = base^0 = 1 for every base, so

    R_p (x, y) = (x cos p - y sin p,  y cos p + x sin p).

For q = (1, 0) at position t:  R_t q = (cos t, sin t)
  key (1, 0) at position a:     R_a k = (cos a, sin a)   -> q.k =  cos(a - t)
  key (0, 1) at position b:     R_b k = (-sin b, cos b)  -> q.k = -sin(b - t)
For q = (0, 1) at position t:  R_t q = (-sin t, cos t)
  key (1, 0) at position a:                              -> q.k =  sin(a - t)
  key (0, 1) at position b:                              -> q.k =  cos(b - t)

Values are v1 = (1, 0) and v2 = (0, 1), so the output is the softmax weight
vector itself, and lse = log(exp(s1) + exp(s2)).  The expected numbers below
are these closed forms evaluated with Python's math module; nothing here calls
the oracle or the CUDA library.  Run:  python tests/golden/make_worked_examples.py
"""

import json
import math
import os

S = 1.0 / math.sqrt(2.0)


def softmax2(s1, s2):
    m = max(s1, s2)
    e1, e2 = math.exp(s1 - m), math.exp(s2 - m)
    z = e1 + e2
    return [e1 / z, e2 / z], m + math.log(z)


def main():
    cases = []
    # Decode, one kv head, two query heads (GQA 2:1).  Keys live in physical
    # blocks 1 and 0 (block size 1) at positions a = 2 and b = 7; query at t = 5.
    t, a, b = 5, 2, 7
    h0 = softmax2(S * math.cos(a - t), S * -math.sin(b - t))
    h1 = softmax2(S * math.sin(a - t), S * math.cos(b - t))
    cases.append({
        "name": "decode_gqa_two_keys",
        "kind": "decode", "Hq": 2, "Hkv": 1, "d": 2, "block_size": 1, "rope_base": 10000.0,
        "q": [[[1.0, 0.0], [0.0, 1.0]]],
        # k_pool/v_pool [num_blocks=2][Hkv=1][bs=1][d=2]; logical key 0 is in block 1
        "k_pool": [[[[0.0, 1.0]]], [[[1.0, 0.0]]]],
        "v_pool": [[[[0.0, 1.0]]], [[[1.0, 0.0]]]],
        "block_tables": [[1, 0]], "block_starts": [[a, b]], "seq_lens": [2], "q_pos": [t],
        "expect_out": [[h0[0], h1[0]]], "expect_lse": [[h0[1], h1[1]]],
        "formula": "head0: s=(cos(a-t), -sin(b-t))/sqrt2; head1: s=(sin(a-t), cos(b-t))/sqrt2",
    })
    # Same keys at a large shared offset: only position differences matter.
    off = 100000
    cases.append(dict(cases[0], name="decode_gqa_two_keys_shifted",
                      block_starts=[[a + off, b + off]], q_pos=[t + off]))
    # Prefill, causal: chunk of 2 queries (positions 6, 7) over its own 2 keys
    # (positions 3, 4).  Query 0 sees key 0 only: out = v1, lse = s1.
    tq = [6, 7]
    pa, pb = 3, 4
    s00 = S * math.cos(pa - tq[0])
    o1, l1 = softmax2(S * math.cos(pa - tq[1]), S * -math.sin(pb - tq[1]))
    cases.append({
        "name": "prefill_causal_two_tokens",
        "kind": "prefill", "Hq": 1, "Hkv": 1, "d": 2, "block_size": 1, "rope_base": 500000.0,
        "q": [[[1.0, 0.0]], [[1.0, 0.0]]],
        "k_pool": [[[[1.0, 0.0]]], [[[0.0, 1.0]]]],
        "v_pool": [[[[1.0, 0.0]]], [[[0.0, 1.0]]]],
        "block_tables": [[0, 1]], "block_starts": [[pa, pb]],
        "cu_q_lens": [0, 2], "q_pos": tq, "kv_lens": [2],
        "expect_out": [[[1.0, 0.0]], [o1]], "expect_lse": [[s00], [l1]],
        "formula": "q0: one key, s=cos(pa-t0)/sqrt2; q1: s=(cos(pa-t1), -sin(pb-t1))/sqrt2",
    })
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "worked_examples.json")
    with open(path, "w") as f:
        json.dump({"source": "MiniPIC summary (gist.science 2606.13126) section 2.1 score equation; "
                             "closed forms for head_dim 2, see make_worked_examples.py",
                   "cases": cases}, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
