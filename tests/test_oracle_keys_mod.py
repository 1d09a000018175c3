"""Pins of the oracle's key-set selection, log-sum-exp combination, adaLN-single
modulation of the attention, and adaLN-single parameters.

Each check compares with something other than the function under test: torch's
float64 scaled_dot_product_attention over independently gathered keys (a library
routine), the identity that two softmaxes over disjoint key sets combined by their
log-sum-exps equal the softmax over the union, closed forms (equal scores give the
mean of the values; a zero modulation changes nothing; a gate scales the output),
and hand-computed adaLN-single outputs for tiny weights.
"""
import numpy as np
import pytest
import torch

import oracle
from block_mask_diffusion_tt_b300 import synth


def _inputs(B=3, S=4, Hq=4, Hkv=2, d=16, Lmax=20, lens=(20, 7, 0), seed=1):
    return synth.attn_inputs(synth.AttnShape(B, S, Hq, Hkv, d, Lmax, lens=list(lens)), seed=seed)


def _sdpa(q, k, v):
    """torch float64 SDPA for one (b): q [S,Hq,d], k/v [n,Hkv,d] (GQA by repetition)."""
    S, Hq, d = q.shape
    G = Hq // k.shape[1]
    qq = torch.from_numpy(q).permute(1, 0, 2)[None]
    kk = torch.from_numpy(np.repeat(k, G, axis=1)).permute(1, 0, 2)[None]
    vv = torch.from_numpy(np.repeat(v, G, axis=1)).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qq, kk, vv)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("keys", ["prefix", "block"])
def test_key_sets_equal_library_attention_over_gathered_keys(keys):
    inp = _inputs()
    out, lse = oracle.block_attn(inp["q"], inp["k_ctx"], inp["v_ctx"], inp["ctx_lens"],
                                 inp["k_blk"], inp["v_blk"], keys=keys)
    dec = oracle.bf16_decode
    for b in range(3):
        L = int(inp["ctx_lens"][b])
        if keys == "prefix":
            k = dec(inp["k_ctx"][b, :, :L]).transpose(1, 0, 2)
            v = dec(inp["v_ctx"][b, :, :L]).transpose(1, 0, 2)
        else:
            k, v = dec(inp["k_blk"][b]), dec(inp["v_blk"][b])
        if k.shape[0] == 0:  # a prefix that is empty: no key at all
            assert (out[b] == 0).all() and np.isneginf(lse[b]).all()
            continue
        np.testing.assert_allclose(out[b], _sdpa(dec(inp["q"][b]), k, v), atol=1e-12)


def test_combined_key_sets_equal_the_one_softmax():
    inp = _inputs()
    args = (inp["q"], inp["k_ctx"], inp["v_ctx"], inp["ctx_lens"], inp["k_blk"], inp["v_blk"])
    full, full_lse = oracle.block_attn(*args)
    o1, l1 = oracle.block_attn(*args, keys="prefix")
    o2, l2 = oracle.block_attn(*args, keys="block")
    o, lse = oracle.lse_combine(o1, l1, o2, l2)
    np.testing.assert_allclose(o, full, atol=1e-12)
    np.testing.assert_allclose(lse, full_lse, atol=1e-12)
    # a side without keys weighs nothing
    o, lse = oracle.lse_combine(o2, l2, np.zeros_like(o2), np.full_like(l2, -np.inf))
    np.testing.assert_allclose(o, o2, atol=0)
    np.testing.assert_allclose(lse, l2, atol=0)


def test_zero_modulation_changes_nothing_and_gate_scales():
    inp = _inputs()
    args = (inp["q"], inp["k_ctx"], inp["v_ctx"], inp["ctx_lens"], inp["k_blk"], inp["v_blk"])
    base, base_lse = oracle.block_attn(*args)
    z = np.zeros((3, 4, 16))
    out, lse = oracle.block_attn(*args, q_scale=z, q_shift=z, o_gate=np.ones((3, 4, 16)))
    np.testing.assert_allclose(out, base, atol=1e-15)
    np.testing.assert_allclose(lse, base_lse, atol=1e-15)
    g = np.random.default_rng(2).uniform(-2, 2, (3, 4, 16))
    out, _ = oracle.block_attn(*args, o_gate=g)
    np.testing.assert_allclose(out, base * g[:, None], atol=1e-14)


def test_scale_minus_one_gives_equal_scores():
    """q (1 + (-1)) + 0 = 0 for every query: all scores equal, so the output is the
    mean of the visible values (closed form)."""
    inp = _inputs()
    z = np.zeros((3, 4, 16))
    out, _ = oracle.block_attn(inp["q"], inp["k_ctx"], inp["v_ctx"], inp["ctx_lens"],
                               inp["k_blk"], inp["v_blk"], q_scale=-np.ones((3, 4, 16)), q_shift=z)
    dec = oracle.bf16_decode
    for b in range(3):
        L = int(inp["ctx_lens"][b])
        vals = np.concatenate([dec(inp["v_ctx"][b, :, :L]).transpose(1, 0, 2),
                               dec(inp["v_blk"][b])], axis=0)  # [n, Hkv, d]
        mean = vals.mean(axis=0)  # [Hkv, d]
        for h in range(4):
            np.testing.assert_allclose(out[b, :, h], np.broadcast_to(mean[h // 2], (4, 16)),
                                       atol=1e-12)


def test_adaln_single_closed_forms():
    """F = 4 (frequencies 1 and 1/100), Dh = 4, W1 = I, b1 = 0, W2 stacking three
    identities, b2 = 0: shift = scale = gate = SiLU(e(t)) + embed[layer] parts."""
    F, Dh, N = 4, 4, 4
    t = np.array([0.0, 1.0, 2.5])
    embed = np.arange(2 * 3 * N, dtype=np.float64).reshape(2, 3 * N) / 10.0
    w2 = np.concatenate([np.eye(N)] * 3, axis=0)
    sh, sc, gt = oracle.adaln_single(t, np.eye(Dh, F), np.zeros(Dh), w2, np.zeros(3 * N), embed, 1)
    for i, tv in enumerate(t):
        e = np.array([np.cos(tv), np.cos(tv / 100.0), np.sin(tv), np.sin(tv / 100.0)])
        silu = e / (1.0 + np.exp(-e))
        np.testing.assert_allclose(sh[i], silu + embed[1, :N], atol=1e-15)
        np.testing.assert_allclose(sc[i], silu + embed[1, N:2 * N], atol=1e-15)
        np.testing.assert_allclose(gt[i], silu + embed[1, 2 * N:], atol=1e-15)
    # zero weights: the per-layer offset alone
    sh, sc, gt = oracle.adaln_single(t, np.zeros((Dh, F)), np.zeros(Dh), np.zeros((3 * N, Dh)),
                                     np.zeros(3 * N), embed, 0)
    assert np.array_equal(np.concatenate([sh, sc, gt], axis=1), np.broadcast_to(embed[0], (3, 3 * N)))
