"""Pins of the oracle's block-by-block generation (oracle.generate_blocks).

Each expected value below is derived from the definition by hand, not by calling
the function under test another way: the number of blocks, the generated lengths
with and without EOS, the steps a block takes when exactly one position commits per
step, and the context cache rebuilt by concatenating the prefix and the appended
blocks.  Block-by-block generation follows the two-tower mechanism of the
dothoosh.com article and the generate call of the 889990.xyz code example
(max_new_tokens, block_size, steps_per_block, eos_token_id).
"""
import numpy as np
import pytest

import oracle

V, MASK = 40, 3


def _logits_fn(seed, B, S, eos=None, eos_at=None):
    """Random fp32 logits per (block, step); eos_at = {(block, b): s} plants a dominant
    EOS at position s of that block (and keeps EOS low everywhere else)."""
    def fn(block, step):
        rng = np.random.default_rng([seed, block, step])
        lg = rng.standard_normal((B, S, V)).astype(np.float32)
        if eos is not None:
            lg[:, :, eos] = -30.0
            for (blk, b), s in (eos_at or {}).items():
                if blk == block:
                    lg[b, s, eos] = 60.0
        return lg
    return fn


def _kv_fn(B, S, Hkv, d, layers):
    """K/V of block `block`: every element equals block + 1 (K) or -(block + 1) (V)
    plus a per-(b, s) offset, so rows can be recognised in the cache."""
    def fn(block, tokens):
        base = (np.arange(B)[:, None] * 100 + np.arange(S)[None, :]).astype(np.float32)
        k = [np.broadcast_to((block + 1) * 1000 + base[:, :, None, None],
                             (B, S, Hkv, d)).astype(np.float32).copy() for _ in range(layers)]
        v = [-x for x in k]
        return k, v
    return fn


def _caches(B, Hkv, Lmax, d, layers, lens):
    k = [np.zeros((B, Hkv, Lmax, d), np.float32) for _ in range(layers)]
    v = [np.zeros((B, Hkv, Lmax, d), np.float32) for _ in range(layers)]
    for layer in range(layers):
        for b in range(B):
            k[layer][b, :, :lens[b]] = 7.0  # the prefix
            v[layer][b, :, :lens[b]] = -7.0
    return k, v


def _run(B=3, S=4, Hkv=2, d=8, layers=2, Lmax=64, lens=(5, 0, 9), max_new=12, eos=-1,
         eos_at=None, gamma=1.5, steps=None, active=None, seed=0):
    k, v = _caches(B, Hkv, Lmax, d, layers, lens)
    return oracle.generate_blocks(
        B, S, _logits_fn(seed, B, S, eos if eos >= 0 else None, eos_at),
        _kv_fn(B, S, Hkv, d, layers), k, v, np.array(lens, np.int32), "f32", 1.0, gamma, MASK,
        steps or S, max_new, eos, active=active)


def test_blocks_lengths_and_steps_without_eos():
    """max_new = 3 S: three blocks; with gamma > 1 each block commits one position per
    step, so it takes exactly S steps; the prefix grows by S after each block but the
    last."""
    B, S = 3, 4
    r = _run(max_new=3 * S)
    assert r["blocks_run"] == 3
    assert r["gen_len"].tolist() == [3 * S] * B
    assert r["steps_total"].tolist() == [3 * S] * B
    assert r["ctx_lens"].tolist() == [5 + 2 * S, 0 + 2 * S, 9 + 2 * S]
    assert not r["active"].any() and r["overflow"] == 0
    assert (r["out_tokens"] >= 0).all() and (r["out_tokens"] < V).all()


def test_cache_holds_prefix_then_blocks_in_order():
    """Rebuild every cache row by hand: prefix rows, then block j's rows (value
    (j+1)*1000 + 100 b + s) for the appended blocks, zeros after."""
    B, S, Hkv, d, layers, Lmax = 3, 4, 2, 8, 2, 64
    lens = (5, 0, 9)
    r = _run(B, S, Hkv, d, layers, Lmax, lens, max_new=3 * S)
    for layer in range(layers):
        for b in range(B):
            want = np.zeros((Lmax,), np.float32)
            want[:lens[b]] = 7.0
            for j in range(2):  # blocks 0 and 1 are appended, block 2 is the last
                for s in range(S):
                    want[lens[b] + j * S + s] = (j + 1) * 1000 + 100 * b + s
            for g in range(Hkv):
                assert np.array_equal(r["k_ctx"][layer][b, g, :, 0], want)
                assert np.array_equal(r["v_ctx"][layer][b, g, :, 0], -want)


def test_eos_stops_only_its_sequence():
    """EOS committed at position 2 of block 1 by sequence 1: its length is 1*S + 2 + 1,
    it takes no part in block 2 and nothing more is appended for it; the others run
    to max_new."""
    B, S, eos = 3, 4, 9
    r = _run(max_new=3 * S, eos=eos, eos_at={(1, 1): 2}, gamma=0.0)
    assert r["gen_len"].tolist() == [3 * S, S + 3, 3 * S]
    assert r["out_tokens"][1, S + 2] == eos
    assert (r["out_tokens"][1, 2 * S:] == -1).all()  # block 2 not generated for it
    assert r["ctx_lens"].tolist() == [5 + 2 * S, 0 + S, 9 + 2 * S]
    assert r["blocks_run"] == 3


def test_eos_in_the_first_block_of_every_sequence_ends_generation():
    B, S, eos = 3, 4, 9
    r = _run(max_new=5 * S, eos=eos, eos_at={(0, 0): 0, (0, 1): 3, (0, 2): 1}, gamma=0.0)
    assert r["blocks_run"] == 1
    assert r["gen_len"].tolist() == [1, 4, 2]
    assert r["ctx_lens"].tolist() == [5, 0, 9]  # nothing appended


def test_max_new_not_a_multiple_of_the_block():
    """max_new = 2 S + 1: three blocks run, one position of the last is kept."""
    B, S = 3, 4
    r = _run(max_new=2 * S + 1)
    assert r["blocks_run"] == 3
    assert r["gen_len"].tolist() == [2 * S + 1] * B
    assert r["out_tokens"].shape == (B, 2 * S + 1)


def test_cache_capacity_stops_a_sequence():
    """Lmax = 14, S = 4, four blocks.  Sequence 2 (prefix 9) takes block 0 into its
    cache (13) but not block 1 (17 > 14): it stops after its second block.  Sequence 0
    (prefix 5) takes blocks 0 and 1 (13) but not block 2: it stops after its third.
    Sequence 1 (prefix 0) runs to max_new.  Two stops are counted as overflow."""
    S = 4
    r = _run(Lmax=14, lens=(5, 0, 9), max_new=4 * S)
    assert r["gen_len"].tolist() == [3 * S, 4 * S, 2 * S]
    assert r["overflow"] == 2
    assert r["ctx_lens"].tolist() == [5 + 2 * S, 0 + 3 * S, 9 + S]


def test_inactive_sequence_is_untouched():
    S = 4
    r = _run(max_new=2 * S, active=np.array([1, 0, 1], np.uint8))
    assert r["gen_len"][1] == 0 and (r["out_tokens"][1] == -1).all()
    assert r["ctx_lens"][1] == 0 and r["steps_total"][1] == 0


def test_planted_mistake_in_eos_rule_is_caught():
    """A generate that ignored EOS would give sequence 1 the full length: the pin above
    would see 3 S where the definition gives S + 3."""
    B, S, eos = 3, 4, 9
    r = _run(max_new=3 * S, eos=-1, eos_at={(1, 1): 2}, gamma=0.0)  # EOS id not passed
    assert r["gen_len"][1] == 3 * S != S + 3
