"""Pins of the fp64 oracle against facts other than itself.

Each ``check_*`` takes a loaded oracle library handle and raises AssertionError
when the oracle disagrees with a closed form, an invariant, a library special
case (torch's scaled_dot_product_attention, scipy's softmax/logsumexp, numpy's
first-occurrence argmax) or a hand-derived worked example.  The same checks run
against deliberately broken copies of the oracle (test_oracle_mutants.py) to show
that each plausible mistake is caught by at least one of them.
"""
from __future__ import annotations

import math
import os

import numpy as np
import scipy.special
import torch

import oracle
from block_mask_diffusion_tt_b300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = [float(v) for v in vals]
    return out


def bf16_exact(x) -> np.ndarray:
    """bf16 bits of values that bf16 represents exactly (asserted)."""
    x = np.asarray(x, dtype=np.float32)
    bits = synth.bf16_bits(x)
    assert np.array_equal(synth.bf16_to_f32(bits), x), "value not exact in bf16"
    return bits


def f64(bits) -> np.ndarray:
    return synth.bf16_to_f32(bits).astype(np.float64)


# ------------------------------------------------------------------ attention
def sdpa_reference(inp, scale=None):
    """torch float64 scaled_dot_product_attention over prefix ++ block keys, per sequence."""
    q, kc, vc, kb, vb, lens = (inp[k] for k in ("q", "k_ctx", "v_ctx", "k_blk", "v_blk", "ctx_lens"))
    B, S, Hq, d = q.shape
    Hkv = kc.shape[1]
    G = Hq // Hkv
    out = np.empty((B, S, Hq, d))
    lse = np.empty((B, Hq, S))
    for b in range(B):
        L = int(lens[b])
        keys = np.concatenate([f64(kc[b, :, :L, :]), f64(kb[b]).transpose(1, 0, 2)], axis=1)
        vals = np.concatenate([f64(vc[b, :, :L, :]), f64(vb[b]).transpose(1, 0, 2)], axis=1)
        qt = torch.from_numpy(f64(q[b]).transpose(1, 0, 2).copy())[None]  # [1,Hq,S,d]
        kt = torch.from_numpy(keys).repeat_interleave(G, dim=0)[None]
        vt = torch.from_numpy(vals).repeat_interleave(G, dim=0)[None]
        sc = 1.0 / math.sqrt(d) if scale is None else scale
        o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=sc)
        out[b] = o[0].numpy().transpose(1, 0, 2)
        scores = torch.einsum("hsd,hjd->hsj", qt[0], kt[0]).numpy() * sc
        lse[b] = scipy.special.logsumexp(scores, axis=-1)
    return out, lse


def run_attn(lib, inp, scale=0.0):
    return oracle.block_attn(inp["q"], inp["k_ctx"], inp["v_ctx"], inp["ctx_lens"], inp["k_blk"],
                             inp["v_blk"], scale=scale, lib=lib)


def check_attn_golden_two_keys(lib):
    g = read_golden("attn_two_keys.txt")
    inp = dict(q=bf16_exact([[[g["q"]]]]), k_ctx=bf16_exact([[[g["k0"]]]]),
               v_ctx=bf16_exact([[[g["v0"]]]]), k_blk=bf16_exact([[[g["k1"]]]]),
               v_blk=bf16_exact([[[g["v1"]]]]), ctx_lens=np.array([1], np.int32))
    out, lse = run_attn(lib, inp, scale=g["scale"][0])
    np.testing.assert_allclose(out[0, 0, 0], g["out"], rtol=1e-14, atol=0)
    np.testing.assert_allclose(lse[0, 0, 0], g["lse"][0], rtol=1e-14, atol=0)


def check_attn_single_key_returns_value(lib):
    inp = synth.attn_inputs(synth.AttnShape(2, 1, 4, 2, 64, 8, lens=[0, 0]), seed=11)
    out, lse = run_attn(lib, inp)
    expect = np.repeat(f64(inp["v_blk"][:, 0]), 2, axis=1)  # [B,Hq,d], GQA groups of 2
    assert np.array_equal(out[:, 0], expect)
    assert np.allclose(lse[:, :, 0], np.einsum("bhd,bhd->bh", f64(inp["q"][:, 0]),
                                               np.repeat(f64(inp["k_blk"][:, 0]), 2, axis=1))
                       / 8.0, rtol=1e-13, atol=1e-13)


def check_attn_equal_scores_mean(lib):
    inp = synth.attn_inputs(synth.AttnShape(3, 5, 4, 2, 64, 40, lens=[40, 7, 0]), seed=12)
    inp["q"][:] = 0
    out, lse = run_attn(lib, inp)
    for b, L in enumerate(inp["ctx_lens"]):
        for h in range(4):
            g = h // 2
            vals = np.concatenate([f64(inp["v_ctx"][b, g, :L]), f64(inp["v_blk"][b, :, g])], axis=0)
            np.testing.assert_allclose(out[b, :, h], np.broadcast_to(vals.mean(axis=0), (5, 64)),
                                       rtol=1e-12, atol=1e-14)
            np.testing.assert_allclose(lse[b, h], math.log(L + 5), rtol=1e-13)


def check_attn_zero_context_is_block_bidirectional(lib):
    inp = synth.attn_inputs(synth.AttnShape(2, 16, 8, 2, 64, 32, lens=[0, 0]), seed=13, nan_pad=True)
    out, lse = run_attn(lib, inp)
    ref, ref_lse = sdpa_reference(inp)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def check_attn_matches_library_sdpa(lib):
    inp = synth.attn_inputs(synth.AttnShape(3, 6, 8, 2, 64, 50, lens=[50, 17, 1]), seed=14)
    out, lse = run_attn(lib, inp)
    ref, ref_lse = sdpa_reference(inp)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def check_attn_tiny_config_matches_library(lib):
    w = synth.workloads()["tiny"]
    inp = synth.attn_inputs(w.attn, seed=w.seed)
    out, lse = run_attn(lib, inp)
    ref, ref_lse = sdpa_reference(inp)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-12)


def check_attn_explicit_scale(lib):
    inp = synth.attn_inputs(synth.AttnShape(1, 4, 2, 1, 64, 9), seed=15)
    out, _ = run_attn(lib, inp, scale=0.37)
    ref, _ = sdpa_reference(inp, scale=0.37)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)


def check_attn_gqa_equals_repeated_heads(lib):
    inp = synth.attn_inputs(synth.AttnShape(2, 4, 8, 2, 64, 12, lens=[12, 5]), seed=16)
    out, lse = run_attn(lib, inp)
    rep = dict(inp)
    rep["k_ctx"] = np.repeat(inp["k_ctx"], 4, axis=1)
    rep["v_ctx"] = np.repeat(inp["v_ctx"], 4, axis=1)
    rep["k_blk"] = np.repeat(inp["k_blk"], 4, axis=2)
    rep["v_blk"] = np.repeat(inp["v_blk"], 4, axis=2)
    out2, lse2 = run_attn(lib, rep)
    assert np.array_equal(out, out2) and np.array_equal(lse, lse2)


def check_attn_padding_is_never_read(lib):
    shape = synth.AttnShape(3, 4, 4, 2, 64, 24, lens=[24, 3, 0])
    clean = synth.attn_inputs(shape, seed=17)
    poisoned = synth.attn_inputs(shape, seed=17, nan_pad=True)
    out, lse = run_attn(lib, clean)
    out2, lse2 = run_attn(lib, poisoned)
    assert np.isfinite(out2).all() and np.array_equal(out, out2) and np.array_equal(lse, lse2)


def check_attn_prefix_permutation_invariant(lib):
    inp = synth.attn_inputs(synth.AttnShape(1, 3, 4, 2, 64, 30, lens=[30]), seed=18)
    out, lse = run_attn(lib, inp)
    perm = np.random.default_rng(0).permutation(30)
    p = dict(inp)
    p["k_ctx"] = inp["k_ctx"][:, :, perm].copy()
    p["v_ctx"] = inp["v_ctx"][:, :, perm].copy()
    out2, lse2 = run_attn(lib, p)
    np.testing.assert_allclose(out, out2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, rtol=1e-13)


def check_attn_value_shift_equivariant(lib):
    """Weights sum to one: adding a constant vector to every value shifts the output by it."""
    rng = np.random.default_rng(1)
    shape = synth.AttnShape(2, 3, 4, 2, 64, 10, lens=[10, 4])
    inp = synth.attn_inputs(shape, seed=19)
    for key in ("v_ctx", "v_blk"):  # small integers: exact in bf16 before and after the shift
        inp[key] = bf16_exact(rng.integers(-8, 9, size=inp[key].shape))
    c = rng.integers(-8, 9, size=64)
    sh = dict(inp)
    sh["v_ctx"] = bf16_exact(f64(inp["v_ctx"]) + c)
    sh["v_blk"] = bf16_exact(f64(inp["v_blk"]) + c)
    out, _ = run_attn(lib, inp)
    out2, _ = run_attn(lib, sh)
    np.testing.assert_allclose(out2 - out, np.broadcast_to(c, out.shape), rtol=0, atol=1e-12)


def check_attn_key_shift_invariant(lib):
    """A constant added to every key moves each row's scores by one constant."""
    rng = np.random.default_rng(2)
    shape = synth.AttnShape(1, 4, 2, 1, 64, 6)
    inp = synth.attn_inputs(shape, seed=20)
    for key in ("k_ctx", "k_blk"):
        inp[key] = bf16_exact(rng.integers(-8, 9, size=inp[key].shape) / 8.0)
    c = rng.integers(-8, 9, size=64) / 8.0
    sh = dict(inp)
    sh["k_ctx"] = bf16_exact(f64(inp["k_ctx"]) + c)
    sh["k_blk"] = bf16_exact(f64(inp["k_blk"]) + c)
    out, _ = run_attn(lib, inp)
    out2, _ = run_attn(lib, sh)
    np.testing.assert_allclose(out, out2, rtol=1e-10, atol=1e-12)


ATTN_CHECKS = [check_attn_golden_two_keys, check_attn_single_key_returns_value,
               check_attn_equal_scores_mean, check_attn_zero_context_is_block_bidirectional,
               check_attn_matches_library_sdpa, check_attn_tiny_config_matches_library,
               check_attn_explicit_scale, check_attn_gqa_equals_repeated_heads,
               check_attn_padding_is_never_read, check_attn_prefix_permutation_invariant,
               check_attn_value_shift_equivariant, check_attn_key_shift_invariant]


# ------------------------------------------------------------------ unmasking
def unmask(lib, logits, T, gamma, tokens=None, masked=None, force=False, dtype="f32", mask_id=3):
    logits = np.asarray(logits)
    B, S, _ = logits.shape
    tokens = np.full((B, S), mask_id, np.int32) if tokens is None else tokens
    masked = np.ones((B, S), np.uint8) if masked is None else masked
    return oracle.confidence_unmask(logits, dtype, T, gamma, mask_id, tokens, masked,
                                    force_commit_all=force, lib=lib)


def check_unmask_golden_tie_row(lib):
    g = read_golden("unmask_tie_row.txt")
    r = unmask(lib, np.array([[g["logits"]]], np.float32), g["temperature"][0], 2.0)
    assert r["tokens"][0, 0] == int(g["token"][0])
    np.testing.assert_allclose(r["conf"][0, 0], g["conf"][0], rtol=1e-15)


def check_unmask_tokens_and_conf_match_library(lib):
    rng = np.random.default_rng(3)
    logits = (rng.standard_normal((3, 8, 300)) * 2).astype(np.float32)
    logits[0, 0, [5, 9]] = 50.0  # planted ties: lowest index wins
    logits[1, 3, [200, 7, 150]] = 40.0
    logits[2, 5] = 1.25  # an all-equal row
    r = unmask(lib, logits, 0.1, 2.0)  # gamma > 1: single commit, every conf reported
    expect_tok = np.argmax(logits, axis=-1)  # numpy: first occurrence of the maximum
    expect_conf = scipy.special.softmax(logits.astype(np.float64) / 0.1, axis=-1).max(axis=-1)
    assert expect_tok[0, 0] == 5 and expect_tok[1, 3] == 7 and expect_tok[2, 5] == 0
    committed = r["committed_now"] == 1
    assert np.array_equal(r["tokens"][committed], expect_tok[committed])
    np.testing.assert_allclose(r["conf"], expect_conf, rtol=1e-12)
    np.testing.assert_allclose(r["conf"][2, 5], 1.0 / 300, rtol=1e-14)
    # all-masked commit of everything exposes every token
    r_all = unmask(lib, logits, 0.1, 0.0)
    assert np.array_equal(r_all["tokens"], expect_tok)


def check_unmask_single_spike_closed_form(lib):
    V, T = 1000, 0.1
    for a in (0.05, 0.3, 1.0, 2.5):
        logits = np.zeros((1, 2, V), np.float32)
        logits[0, 0, 417] = a
        logits[0, 1, 3] = -a
        r = unmask(lib, logits, T, 0.0)
        a = float(np.float32(a))  # the logit as stored
        assert r["tokens"][0, 0] == 417 and r["tokens"][0, 1] == 0
        np.testing.assert_allclose(r["conf"][0, 0], 1.0 / (1.0 + (V - 1) * math.exp(-a / T)),
                                   rtol=1e-13)
        np.testing.assert_allclose(r["conf"][0, 1], 1.0 / (V - 1 + math.exp(-a / T)), rtol=1e-13)


def check_unmask_gamma_zero_commits_all(lib):
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((2, 16, 64)).astype(np.float32)
    r = unmask(lib, logits, 0.1, 0.0)
    assert r["committed_now"].all() and not r["is_masked"].any() and (r["remaining"] == 0).all()


def check_unmask_gamma_above_one_commits_most_confident(lib):
    rng = np.random.default_rng(5)
    logits = rng.standard_normal((3, 16, 64)).astype(np.float32) * 3
    masked = np.ones((3, 16), np.uint8)
    masked[1, :5] = 0
    tokens = np.full((3, 16), 3, np.int32)
    tokens[1, :5] = 77
    r = unmask(lib, logits, 0.1, 1.5, tokens=tokens, masked=masked)
    expect_conf = scipy.special.softmax(logits.astype(np.float64) / 0.1, axis=-1).max(axis=-1)
    assert (r["committed_now"].sum(axis=1) == 1).all()
    for b in range(3):
        # the decision is taken on fp32 confidences, lowest position on ties
        cand = np.where(masked[b] == 1, expect_conf[b].astype(np.float32), np.float32(-1))
        assert r["committed_now"][b, int(np.argmax(cand))] == 1
    assert np.array_equal(r["tokens"][1, :5], np.full(5, 77))  # committed earlier: untouched
    assert np.isnan(r["conf"][1, :5]).all()
    assert np.array_equal(r["remaining"], np.array([15, 10, 15]))


def check_unmask_threshold_is_inclusive(lib):
    logits = np.zeros((1, 3, 2), np.float32)
    logits[0, 1] = [0.0, -np.inf]  # conf exactly 1
    logits[0, 2] = [-np.inf, 0.0]
    r = unmask(lib, logits, 1.0, 0.5)  # row 0: conf exactly 0.5 == gamma commits
    assert r["committed_now"].tolist() == [[1, 1, 1]]
    assert r["tokens"].tolist() == [[0, 0, 1]]
    r2 = unmask(lib, logits, 1.0, np.nextafter(np.float32(0.5), np.float32(1)))
    assert r2["committed_now"].tolist() == [[0, 1, 1]]


def check_unmask_fallback_ties_to_lowest_position(lib):
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((1, 8, 50)).astype(np.float32) * 0.01  # flat: conf ~ 1/50
    logits[0, 2, 10] = logits[0, 5, 10] = 0.2  # s=2 and s=5 identical, most confident
    logits[0, 5] = logits[0, 2]
    r = unmask(lib, logits, 0.1, 0.9)
    assert r["committed_now"][0].tolist() == [0, 0, 1, 0, 0, 0, 0, 0]
    assert r["tokens"][0, 2] == 10 and r["remaining"][0] == 7


def check_unmask_remasks_uncommitted(lib):
    logits = np.zeros((1, 4, 8), np.float32)
    logits[0, 0, 6] = 20.0
    tokens = np.array([[9, 9, 9, 9]], np.int32)  # stale values in masked slots
    r = unmask(lib, logits, 0.1, 0.9, tokens=tokens, mask_id=3)
    assert r["tokens"].tolist() == [[6, 3, 3, 3]]
    assert r["is_masked"].tolist() == [[0, 1, 1, 1]]


def check_unmask_force_commits_everything(lib):
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((2, 6, 30)).astype(np.float32)
    masked = np.array([[1, 0, 1, 1, 0, 1], [0, 0, 0, 0, 0, 0]], np.uint8)
    r = unmask(lib, logits, 0.1, 0.99, masked=masked, force=True)
    assert np.array_equal(r["committed_now"], masked) and (r["remaining"] == 0).all()
    assert np.array_equal(r["tokens"][masked == 1], np.argmax(logits, axis=-1)[masked == 1])


def check_unmask_sequences_independent(lib):
    rng = np.random.default_rng(8)
    logits = rng.standard_normal((3, 8, 40)).astype(np.float32) * 2
    r = unmask(lib, logits, 0.1, 0.8)
    for b in range(3):
        rb = unmask(lib, logits[b:b + 1], 0.1, 0.8)
        for k in ("tokens", "committed_now", "is_masked"):
            assert np.array_equal(r[k][b], rb[k][0])


def check_unmask_bf16_equals_f32_of_same_values(lib):
    rng = np.random.default_rng(9)
    bits = synth.bf16_bits(rng.standard_normal((2, 8, 128)).astype(np.float32) * 2)
    r16 = unmask(lib, bits, 0.1, 0.8, dtype="bf16")
    r32 = unmask(lib, synth.bf16_to_f32(bits), 0.1, 0.8, dtype="f32")
    for k in ("tokens", "committed_now", "is_masked", "remaining"):
        assert np.array_equal(r16[k], r32[k])
    assert np.array_equal(r16["conf"], r32["conf"])


def check_unmask_temperature_closed_form(lib):
    logits = np.array([[[1.5, 0.0, -np.inf]]], np.float32)
    for T in (0.1, 0.5, 2.0):
        r = unmask(lib, logits, T, 0.0)
        assert r["tokens"][0, 0] == 0
        np.testing.assert_allclose(r["conf"][0, 0], 1.0 / (1.0 + math.exp(-1.5 / T)), rtol=1e-14)


UNMASK_CHECKS = [check_unmask_golden_tie_row, check_unmask_tokens_and_conf_match_library,
                 check_unmask_single_spike_closed_form, check_unmask_gamma_zero_commits_all,
                 check_unmask_gamma_above_one_commits_most_confident,
                 check_unmask_threshold_is_inclusive, check_unmask_fallback_ties_to_lowest_position,
                 check_unmask_remasks_uncommitted, check_unmask_force_commits_everything,
                 check_unmask_sequences_independent, check_unmask_bf16_equals_f32_of_same_values,
                 check_unmask_temperature_closed_form]


# ------------------------------------------------------------------ block loop
def _loop(lib, B, S, V, gamma, steps, seed=0, sigma=3.0, p=0.0, start_step=0, state=None):
    fn = lambda k: synth.counter_logits(seed, k, B, S, V, sigma, p, dtype="f32")  # noqa: E731
    return oracle.block_loop(B, S, fn, "f32", 0.1, gamma, 3, steps, start_step=start_step,
                             state=state, lib=lib)


def check_loop_defaults_from_pages(lib):
    g = read_golden("generate_defaults.txt")
    S, steps, mask_id = int(g["block_size"][0]), int(g["steps_per_block"][0]), int(g["mask_token_id"][0])
    assert (S, steps, mask_id) == (16, 16, 3)
    T, gamma = g["temperature"][0], g["confidence_threshold"][0]
    fn = lambda k: synth.counter_logits(0, k, 2, S, 256, 3.0, 0.5, dtype="f32")  # noqa: E731
    seen_masked = []

    def probe(k):
        seen_masked.append(k)
        return fn(k)
    r = oracle.block_loop(2, S, probe, "f32", T, gamma, mask_id, steps, lib=lib)
    assert not r["is_masked"].any()
    assert (r["committed_step"] >= 0).all() and (r["committed_step"] < steps).all()
    assert (r["steps_used"] == r["committed_step"].max(axis=1) + 1).all()
    assert len(seen_masked) == r["steps_used"].max()


def check_loop_gamma_zero_one_step(lib):
    r = _loop(lib, 3, 16, 128, 0.0, 16)
    assert (r["steps_used"] == 1).all() and (r["committed_step"] == 0).all()


def check_loop_gamma_above_one_s_steps(lib):
    S = 8
    r = _loop(lib, 2, S, 128, 1.5, S)
    assert (r["steps_used"] == S).all() and not r["is_masked"].any()
    for b in range(2):
        assert sorted(r["committed_step"][b].tolist()) == list(range(S))
    # S-1 unforced steps commit one position each and leave exactly one masked
    tokens = np.full((2, S), 3, np.int32)
    masked = np.ones((2, S), np.uint8)
    for k in range(S - 1):
        st = unmask(lib, synth.counter_logits(0, k, 2, S, 128, 3.0, dtype="f32"), 0.1, 1.5,
                    tokens=tokens, masked=masked)
        assert (st["committed_now"].sum(axis=1) == 1).all()
        tokens, masked = st["tokens"], st["is_masked"]
    assert (masked.sum(axis=1) == 1).all()


def check_loop_last_step_forces_commit(lib):
    S = 8
    r = _loop(lib, 2, S, 128, 1.5, 3)  # 3 steps for 8 positions: step 2 commits the rest
    assert not r["is_masked"].any() and (r["steps_used"] == 3).all()
    assert ((r["committed_step"] == 2).sum(axis=1) == S - 2).all()


def check_loop_monotone_and_complete(lib):
    B, S, V = 2, 16, 200
    tokens = np.full((B, S), 3, np.int32)
    masked = np.ones((B, S), np.uint8)
    total = np.zeros((B,), np.int64)
    for k in range(S):
        logits = synth.counter_logits(0, k, B, S, V, 3.0, 0.3, dtype="f32")
        r = unmask(lib, logits, 0.1, 0.8, tokens=tokens, masked=masked, force=(k == S - 1))
        was = masked == 0
        assert np.array_equal(r["tokens"][was], tokens[was])  # committed tokens never change
        assert not (r["is_masked"] > masked).any()
        assert np.array_equal(r["tokens"][r["is_masked"] == 1],
                              np.full(int(r["is_masked"].sum()), 3))
        total += r["committed_now"].sum(axis=1).astype(np.int64)
        tokens, masked = r["tokens"], r["is_masked"]
    assert (total == S).all() and not masked.any()


def check_loop_resume_bit_exact(lib):
    B, S, V = 2, 16, 100
    fn = lambda k: synth.counter_logits(0, k, B, S, V, 0.25, 0.15, dtype="f32")  # noqa: E731
    full = oracle.block_loop(B, S, fn, "f32", 0.1, 0.95, 3, 16, lib=lib)
    first = oracle.block_loop(B, S, fn, "f32", 0.1, 0.95, 3, 16, stop_step=8, lib=lib)
    second = oracle.block_loop(B, S, fn, "f32", 0.1, 0.95, 3, 16, start_step=8, state=first,
                               lib=lib)
    assert first["is_masked"].any()  # the split really falls inside the block
    for k in ("tokens", "is_masked", "steps_used", "committed_step"):
        assert np.array_equal(full[k], second[k]), k


LOOP_CHECKS = [check_loop_defaults_from_pages, check_loop_gamma_zero_one_step,
               check_loop_gamma_above_one_s_steps, check_loop_last_step_forces_commit,
               check_loop_monotone_and_complete, check_loop_resume_bit_exact]

# ------------------------------------------------------------------ block append
def _kv_case(seed, B=3, S=4, Hkv=2, d=8, Lmax=12, lens=(0, 5, 8), layers=2):
    rng = np.random.default_rng(seed)
    bits = lambda shape: synth.bf16_bits(rng.standard_normal(shape).astype(np.float32))  # noqa: E731
    kc = [bits((B, Hkv, Lmax, d)) for _ in range(layers)]
    vc = [bits((B, Hkv, Lmax, d)) for _ in range(layers)]
    kb = [bits((B, S, Hkv, d)) for _ in range(layers)]
    vb = [bits((B, S, Hkv, d)) for _ in range(layers)]
    return kc, vc, np.array(lens, np.int32), kb, vb


def kv_append_then_attend(lib, append_fn=None):
    """A block appended to the context, then the next block attending over it, equals torch
    float64 attention over keys concatenated independently: prefix rows, the appended block's
    rows (head-major), the new block's rows."""
    append_fn = append_fn or oracle.kv_append
    kc, vc, lens, kb, vb = _kv_case(31, lens=(0, 5, 7))
    B, S, Hkv, d = kb[0].shape
    r = append_fn(kc, vc, lens, kb, vb)
    rng = np.random.default_rng(32)
    Hq = 2 * Hkv
    q = synth.bf16_bits(rng.standard_normal((B, S, Hq, d)).astype(np.float32))
    ky = synth.bf16_bits(rng.standard_normal((B, S, Hkv, d)).astype(np.float32))
    vy = synth.bf16_bits(rng.standard_normal((B, S, Hkv, d)).astype(np.float32))
    for layer in range(len(kc)):
        got, _ = oracle.block_attn(q, r["k_ctx"][layer], r["v_ctx"][layer], r["ctx_lens"], ky, vy,
                                   lib=lib)
        for b in range(B):
            L = int(lens[b])
            keys = np.concatenate([f64(kc[layer][b, :, :L, :]),
                                   f64(kb[layer][b]).transpose(1, 0, 2),
                                   f64(ky[b]).transpose(1, 0, 2)], axis=1)
            vals = np.concatenate([f64(vc[layer][b, :, :L, :]),
                                   f64(vb[layer][b]).transpose(1, 0, 2),
                                   f64(vy[b]).transpose(1, 0, 2)], axis=1)
            qt = torch.from_numpy(f64(q[b]).transpose(1, 0, 2).copy())[None]
            kt = torch.from_numpy(keys).repeat_interleave(Hq // Hkv, dim=0)[None]
            vt = torch.from_numpy(vals).repeat_interleave(Hq // Hkv, dim=0)[None]
            want = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt)[0].numpy()
            assert np.abs(got[b] - want.transpose(1, 0, 2)).max() < 1e-9, (layer, b)
    assert r["ctx_lens"].tolist() == [L + S for L in lens.tolist()] and r["overflow"] == 0


def check_kv_append_then_attend_matches_library(lib):
    kv_append_then_attend(lib)


def check_kv_two_appends_equal_one_double_block(lib):
    kc, vc, lens, kb, vb = _kv_case(33, S=3, Lmax=14, lens=(0, 2, 8))
    _, _, _, kb2, vb2 = _kv_case(34, S=3, Lmax=14, lens=(0, 2, 8))
    a = oracle.kv_append(kc, vc, lens, kb, vb)
    a = oracle.kv_append(a["k_ctx"], a["v_ctx"], a["ctx_lens"], kb2, vb2)
    kbb = [np.concatenate([x, y], axis=1) for x, y in zip(kb, kb2)]
    vbb = [np.concatenate([x, y], axis=1) for x, y in zip(vb, vb2)]
    b = oracle.kv_append(kc, vc, lens, kbb, vbb)
    for layer in range(len(kc)):
        assert np.array_equal(a["k_ctx"][layer], b["k_ctx"][layer])
        assert np.array_equal(a["v_ctx"][layer], b["v_ctx"][layer])
    assert np.array_equal(a["ctx_lens"], b["ctx_lens"])


def check_kv_untouched_outside_the_block(lib):
    # lengths 0, 8 (fits exactly: 8 + 4 = Lmax), 9 (does not fit), -1 (invalid), 3 (inactive)
    kc, vc, lens, kb, vb = _kv_case(35, B=5, Lmax=12, lens=(0, 8, 9, -1, 3))
    active = np.array([1, 1, 1, 1, 0], np.uint8)
    r = oracle.kv_append(kc, vc, lens, kb, vb, active=active)
    assert r["overflow"] == 2
    assert r["ctx_lens"].tolist() == [4, 12, 9, -1, 3]
    S = kb[0].shape[1]
    for layer in range(len(kc)):
        for b, L in enumerate(lens.tolist()):
            written = L + S if r["ctx_lens"][b] != L else L
            keep = np.ones(kc[layer].shape[2], bool)
            keep[max(L, 0):written] = False
            assert np.array_equal(r["k_ctx"][layer][b][:, keep], kc[layer][b][:, keep])
            assert np.array_equal(r["v_ctx"][layer][b][:, keep], vc[layer][b][:, keep])


KV_CHECKS = [check_kv_append_then_attend_matches_library, check_kv_two_appends_equal_one_double_block,
             check_kv_untouched_outside_the_block]

ALL_CHECKS = ATTN_CHECKS + UNMASK_CHECKS + LOOP_CHECKS + KV_CHECKS
