"""Pins of the block-hash chain oracle (MiniPIC summary, section 2.2: SSEP
restarts the chain, PDEP makes a block depend on the whole prompt before it)
and of its prefix-cache mapping.  CPU only."""

import numpy as np
import pytest

import oracle.blockhash as bh

BS, SSEP, PDEP, H0 = 4, -7, -9, 0x1234


def test_fnv1a64_published_vectors():
    # the FNV reference test vectors of the 64-bit FNV-1a function
    assert bh.fnv1a64(b"") == 0xCBF29CE484222325
    assert bh.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert bh.fnv1a64(b"foobar") == 0x85944171F73967E8


def test_chain_hash_reads_parent_then_int32_tokens_little_endian():
    # H(parent, tokens) hashes 8 parent bytes then 4 bytes per token, so a
    # chain step equals FNV-1a continued over the token bytes from the state
    # reached after the parent bytes
    state = bh.fnv1a64((0x0102030405060708).to_bytes(8, "little"))
    assert bh.chain_hash(0x0102030405060708, [1, -1]) == bh.fnv1a64(
        b"\x01\x00\x00\x00\xff\xff\xff\xff", state)
    assert bh.chain_hash(5, []) == bh.fnv1a64(b"\x05" + b"\x00" * 7)


def _prompt(prefix, span, suffix):
    return list(prefix) + list(span) + list(suffix)


def test_ssep_span_is_cached_whatever_precedes_it():
    span = [SSEP, 11, 12, 13, 21, 22, 23, 24]          # two blocks
    a = bh.block_hashes(_prompt([1, 2, 3, 4], span, []), BS, SSEP, PDEP, H0)
    b = bh.block_hashes(_prompt([5, 6, 7, 8, 9, 10, 11, 12], span, []), BS, SSEP, PDEP, H0)
    assert a[1:] == b[2:]          # both span blocks match
    assert a[0] != b[0]


def test_default_chain_depends_on_the_prefix():
    span = [31, 11, 12, 13, 21, 22, 23, 24]            # no separator
    a = bh.block_hashes(_prompt([1, 2, 3, 4], span, []), BS, SSEP, PDEP, H0)
    b = bh.block_hashes(_prompt([5, 2, 3, 4], span, []), BS, SSEP, PDEP, H0)
    assert all(x != y for x, y in zip(a, b))
    # ... and equals the chain restarted at the root when nothing precedes it
    c = bh.block_hashes(span, BS, SSEP, PDEP, H0)
    assert c[0] == bh.chain_hash(H0, span[:4]) and c[1] == bh.chain_hash(c[0], span[4:])


def test_pdep_depends_on_the_whole_prompt_across_restarts():
    span = [SSEP, 11, 12, 13]
    tail = [PDEP, 41, 42, 43]
    a = bh.block_hashes(_prompt([1, 2, 3, 4], span, tail), BS, SSEP, PDEP, H0)
    b = bh.block_hashes(_prompt([5, 2, 3, 4], span, tail), BS, SSEP, PDEP, H0)
    assert a[1] == b[1]            # the SSEP span is shared
    assert a[2] != b[2]            # the PDEP block is not: its prompts differ
    whole = _prompt([1, 2, 3, 4], span, tail)
    assert a[2] == bh.chain_hash(H0, whole)
    # without the PDEP token the block would chain from the span and be shared
    c = bh.block_hashes(_prompt([1, 2, 3, 4], span, [40, 41, 42, 43]), BS, SSEP, PDEP, H0)
    d = bh.block_hashes(_prompt([5, 2, 3, 4], span, [40, 41, 42, 43]), BS, SSEP, PDEP, H0)
    assert c[2] == d[2]


def test_only_full_blocks_are_hashed():
    assert len(bh.block_hashes(list(range(11)), BS, SSEP, PDEP, H0)) == 2
    assert bh.block_hashes([], BS, SSEP, PDEP, H0) == []


def test_special_tokens_only_count_at_a_block_start():
    a = bh.block_hashes([1, SSEP, 2, 3, 4, 5, 6, 7], BS, SSEP, PDEP, H0)
    b = bh.block_hashes([9, SSEP, 2, 3, 4, 5, 6, 7], BS, SSEP, PDEP, H0)
    assert a[1] != b[1]            # SSEP inside a block restarts nothing


def test_cache_shares_blocks_at_different_offsets():
    span = [SSEP, 11, 12, 13, 21, 22, 23, 24]
    p1 = _prompt([1, 2, 3, 4], span, [7, 7])             # span at token 4
    p2 = _prompt([5, 6, 7, 8, 9, 10, 11, 12], span, [])  # span at token 8
    c = bh.PrefixCache(16)
    t1, s1, n1 = c.assign(bh.block_hashes(p1, BS, SSEP, PDEP, H0), 4, BS)
    t2, s2, n2 = c.assign(bh.block_hashes(p2, BS, SSEP, PDEP, H0), 4, BS)
    assert list(t1[1:3]) == list(t2[2:4])               # the span's two physical blocks
    assert list(s1[1:3]) == [4, 8] and list(s2[2:4]) == [8, 12]   # at different logical offsets
    assert list(n1) == [1, 1, 1, 1] and list(n2) == [1, 1, 0, 0]
    assert len(set(t1) | set(t2)) == 6


def test_cache_evicts_the_longest_released_block_and_rolls_back_when_full():
    c = bh.PrefixCache(3)
    ha = bh.block_hashes([SSEP, 1, 1, 1], BS, SSEP, PDEP, H0)
    hb = bh.block_hashes([SSEP, 2, 2, 2], BS, SSEP, PDEP, H0)
    hc = bh.block_hashes([SSEP, 3, 3, 3], BS, SSEP, PDEP, H0)
    hd = bh.block_hashes([SSEP, 4, 4, 4], BS, SSEP, PDEP, H0)
    ta = c.assign(ha, 1, BS)[0]
    tb = c.assign(hb, 1, BS)[0]
    tc = c.assign(hc, 1, BS)[0]
    assert c.assign(hd, 1, BS) is None                 # all three referenced
    c.release(tb)
    c.release(ta)
    td, _, nd = c.assign(hd, 1, BS)
    assert td[0] == tb[0] and nd[0] == 1               # b was released first
    assert c.assign(ha, 1, BS)[2][0] == 0              # a still cached: a hit
    assert c.assign(hb, 1, BS) is None                 # b was evicted and nothing is free
    c.release(tc)
    tb2, _, nb2 = c.assign(hb, 1, BS)
    assert nb2[0] == 1 and tb2[0] == tc[0]


_ORIGINAL = bh.block_hashes


def _no_reset(tokens, block_size, ssep, pdep, h0):
    # planted mistake: SSEP does not restart the chain
    return _ORIGINAL(tokens, block_size, object(), pdep, h0)


def _pdep_own_block(tokens, block_size, ssep, pdep, h0):
    # planted mistake: PDEP hashes only its own block
    toks = list(tokens)
    out = _ORIGINAL(toks, block_size, ssep, object(), h0)
    for i in range(len(out)):
        if toks[i * block_size] == pdep:
            out[i] = bh.chain_hash(h0, toks[i * block_size:(i + 1) * block_size])
    return out


@pytest.mark.parametrize("mutant,test", [(_no_reset, test_ssep_span_is_cached_whatever_precedes_it),
                                         (_pdep_own_block, test_pdep_depends_on_the_whole_prompt_across_restarts)])
def test_pins_catch_planted_mistakes(monkeypatch, mutant, test):
    test()
    monkeypatch.setattr(bh, "block_hashes", mutant)
    with pytest.raises(AssertionError):
        test()
