"""GPU parity of tt_block_attn_ex (key sets, paged cache, adaLN-single modulation),
tt_attn_lse_combine and tt_adaln_single against the fp64 oracle.

Tolerances as for tt_block_attn: max-abs 1.5e-2, mean-abs 2e-3 on the bf16 output,
1e-4 on the log-sum-exp.  The paged cache must also give bit for bit the result of
the contiguous cache holding the same keys (the kernel's arithmetic does not depend
on where a tile comes from), and a zero modulation bit for bit the plain call.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from block_mask_diffusion_tt_b300 import synth, tt
import _gpu

pytestmark = pytest.mark.gpu


def _run_ex(inp, **kw):
    d = _gpu.attn_dev(inp)
    B, S, Hq, _ = inp["q"].shape
    lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device=_gpu.DEV)
    out = tt.block_attn_ex(d["q"], d["k_ctx"], d["v_ctx"], d["ctx_lens"], d["k_blk"], d["v_blk"],
                           lse=lse, **kw)
    torch.cuda.synchronize()
    return out, lse


def _np(t):
    return t.float().cpu().numpy().astype(np.float64)


def _check_lse(got, want, what):
    g, w = got.cpu().numpy().astype(np.float64), want
    assert np.array_equal(np.isneginf(g), np.isneginf(w)), what
    fin = np.isfinite(w)
    assert np.abs(g[fin] - w[fin]).max(initial=0) <= _gpu.LSE_ABS, what


SHAPES = [
    synth.AttnShape(4, 16, 32, 2, 128, 3000, lens=[3000, 0, 65, 1200]),
    synth.AttnShape(1, 16, 16, 1, 128, 20000, lens=[20000]),         # split over many CTAs
    synth.AttnShape(3, 7, 12, 3, 64, 300, lens=[300, 1, 0]),
    synth.AttnShape(64, 16, 32, 2, 128, 130, lens=list(range(0, 128, 2))),  # many short pairs
]


@pytest.mark.parametrize("keys", ["prefix", "block"])
@pytest.mark.parametrize("shape", SHAPES, ids=["ragged", "long", "odd", "short"])
def test_key_sets_match_oracle(shape, keys):
    inp = synth.attn_inputs(shape, seed=shape.B + shape.d)
    k = tt.TT_KEYS_PREFIX if keys == "prefix" else tt.TT_KEYS_BLOCK
    out, lse = _run_ex(inp, keys=k)
    ref, ref_lse = oracle.block_attn(inp["q"], inp["k_ctx"], inp["v_ctx"], inp["ctx_lens"],
                                     inp["k_blk"], inp["v_blk"], keys=keys)
    _gpu.assert_attn_close(_np(out), ref, what=f"keys={keys}")
    _check_lse(lse, ref_lse, f"keys={keys} lse")


@pytest.mark.parametrize("shape", SHAPES[:3], ids=["ragged", "long", "odd"])
def test_two_softmaxes_combined_equal_the_one(shape):
    inp = synth.attn_inputs(shape, seed=shape.B + 7)
    o1, l1 = _run_ex(inp, keys=tt.TT_KEYS_PREFIX)
    o2, l2 = _run_ex(inp, keys=tt.TT_KEYS_BLOCK)
    lse = torch.empty_like(l1)
    out = tt.attn_lse_combine(o1, l1, o2, l2, lse_out=lse)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.block_attn(inp["q"], inp["k_ctx"], inp["v_ctx"], inp["ctx_lens"],
                                     inp["k_blk"], inp["v_blk"])
    _gpu.assert_attn_close(_np(out), ref, what="combined")
    _check_lse(lse, ref_lse, "combined lse")
    # the combination kernel alone, against the oracle's combination of the same halves
    want, _ = oracle.lse_combine(_np(o1), l1.cpu().numpy(), _np(o2), l2.cpu().numpy())
    assert np.abs(_np(out) - want).max() <= 2 ** -7  # one bf16 rounding of the result


def _paged(inp, page_seed):
    """The same keys in a shuffled pool of 64-key pages: [n_pages, Hkv, 64, d]."""
    B, Hkv, Lmax, d = inp["k_ctx"].shape
    maxp = -(-Lmax // 64)
    rng = np.random.default_rng(page_seed)
    n_pages = B * maxp + 3
    perm = rng.permutation(n_pages)[:B * maxp].reshape(B, maxp).astype(np.int32)
    pools = []
    for key in ("k_ctx", "v_ctx"):
        pool = np.zeros((n_pages, Hkv, 64, d), np.uint16)
        padded = np.zeros((B, Hkv, maxp * 64, d), np.uint16)
        padded[:, :, :Lmax] = inp[key]
        for b in range(B):
            for j in range(maxp):
                pool[perm[b, j]] = padded[b, :, 64 * j:64 * (j + 1)]
        pools.append(pool)
    # entries past a sequence's length are never read: poison them
    for b in range(B):
        used = -(-int(inp["ctx_lens"][b]) // 64)
        perm[b, used:] = -7
    return pools, perm, n_pages


@pytest.mark.parametrize("shape", [
    synth.AttnShape(4, 16, 32, 2, 128, 64 * 40, lens=[2560, 0, 65, 1200]),
    synth.AttnShape(2, 16, 16, 1, 64, 64 * 100, lens=[6400, 3333]),
    synth.AttnShape(40, 16, 32, 2, 128, 64 * 3, lens=[(7 * i) % 192 for i in range(40)]),
], ids=["ragged", "long-d64", "short"])
def test_paged_cache_bit_exact_and_oracle(shape):
    inp = synth.attn_inputs(shape, seed=31 + shape.B)
    (kp, vp), table, n_pages = _paged(inp, shape.B)
    d = _gpu.attn_dev(inp)
    B, S, Hq, D = inp["q"].shape
    ref_lse = torch.empty((B, Hq, S), dtype=torch.float32, device=_gpu.DEV)
    contiguous = tt.block_attn(d["q"], d["k_ctx"], d["v_ctx"], d["ctx_lens"], d["k_blk"], d["v_blk"],
                               lse=ref_lse)
    lse = torch.empty_like(ref_lse)
    paged = tt.block_attn_ex(d["q"], _gpu.bf16_dev(kp), _gpu.bf16_dev(vp), d["ctx_lens"], d["k_blk"],
                             d["v_blk"], block_table=torch.from_numpy(table).to(_gpu.DEV),
                             n_pages=n_pages, lse=lse)
    torch.cuda.synchronize()
    assert torch.equal(paged.view(torch.int16), contiguous.view(torch.int16))
    assert torch.equal(lse, ref_lse)
    ref, ref_l = oracle.block_attn(inp["q"], inp["k_ctx"], inp["v_ctx"], inp["ctx_lens"],
                                   inp["k_blk"], inp["v_blk"])
    _gpu.assert_attn_close(_np(paged), ref, lse.cpu().numpy(), ref_l, "paged")


def test_paged_cache_bad_page_is_flagged():
    shape = synth.AttnShape(2, 16, 8, 2, 128, 128, lens=[128, 100])
    inp = synth.attn_inputs(shape, seed=5)
    (kp, vp), table, n_pages = _paged(inp, 1)
    table[1, 1] = n_pages + 5  # a page outside the pool, inside sequence 1's length
    d = _gpu.attn_dev(inp)
    desc = tt.attn_desc(d["q"], d["k_ctx"], d["v_ctx"], d["k_blk"], d["v_blk"], d["q"])
    ws = tt.Workspace(tt.block_attn_workspace_size(desc))
    tt.block_attn_ex(d["q"], _gpu.bf16_dev(kp), _gpu.bf16_dev(vp), d["ctx_lens"], d["k_blk"],
                     d["v_blk"], block_table=torch.from_numpy(table).to(_gpu.DEV), n_pages=n_pages,
                     workspace=ws)
    torch.cuda.synchronize()
    flag = ctypes.c_int32(-1)
    tt.check(tt.load().tt_block_attn_error(ws.ptr, ctypes.byref(flag), None))
    assert flag.value == 16


@pytest.mark.parametrize("shape", [
    synth.AttnShape(4, 16, 32, 2, 128, 1500, lens=[1500, 0, 300, 999]),
    synth.AttnShape(1, 16, 16, 1, 128, 20000, lens=[20000]),
    synth.AttnShape(3, 5, 8, 2, 64, 200, lens=[200, 1, 77]),
], ids=["ragged", "long", "d64"])
def test_modulation_matches_oracle(shape):
    inp = synth.attn_inputs(shape, seed=41 + shape.B)
    B, S, Hq, D = inp["q"].shape
    rng = np.random.default_rng(B)
    sc = rng.uniform(-0.5, 0.5, (B, Hq, D)).astype(np.float32)
    sh = rng.uniform(-0.5, 0.5, (B, Hq, D)).astype(np.float32)
    gt = rng.uniform(-1.5, 1.5, (B, Hq, D)).astype(np.float32)
    dev = lambda x: torch.from_numpy(x).to(_gpu.DEV)  # noqa: E731
    out, lse = _run_ex(inp, q_scale=dev(sc), q_shift=dev(sh), o_gate=dev(gt))
    ref, ref_lse = oracle.block_attn(inp["q"], inp["k_ctx"], inp["v_ctx"], inp["ctx_lens"],
                                     inp["k_blk"], inp["v_blk"], q_scale=sc, q_shift=sh, o_gate=gt)
    # the kernel rounds the modulated queries to bf16 before the scores; the scores then
    # differ from the fp64 oracle's by up to |q'| 2^-9 |k| scale, within the tolerance
    _gpu.assert_attn_close(_np(out), ref, what="modulated")
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= 2e-2


def test_zero_modulation_is_the_plain_call():
    shape = synth.AttnShape(4, 16, 32, 2, 128, 1500, lens=[1500, 0, 300, 999])
    inp = synth.attn_inputs(shape, seed=9)
    d = _gpu.attn_dev(inp)
    B, S, Hq, D = inp["q"].shape
    plain = tt.block_attn(d["q"], d["k_ctx"], d["v_ctx"], d["ctx_lens"], d["k_blk"], d["v_blk"])
    z = torch.zeros((B, Hq, D), dtype=torch.float32, device=_gpu.DEV)
    one = torch.ones_like(z)
    mod = tt.block_attn_ex(d["q"], d["k_ctx"], d["v_ctx"], d["ctx_lens"], d["k_blk"], d["v_blk"],
                           q_scale=z, q_shift=z, o_gate=one)
    torch.cuda.synchronize()
    assert torch.equal(mod.view(torch.int16), plain.view(torch.int16))


def test_adaln_single_matches_oracle():
    rng = np.random.default_rng(12)
    B, F, Dh, N, layers = 32, 256, 128, 32 * 128, 6
    t = rng.uniform(0, 1, B).astype(np.float32)
    w1 = (rng.standard_normal((Dh, F)) / np.sqrt(F)).astype(np.float32)
    b1 = (rng.standard_normal(Dh) * 0.1).astype(np.float32)
    w2 = (rng.standard_normal((3 * N, Dh)) / np.sqrt(Dh) * 0.1).astype(np.float32)
    b2 = (rng.standard_normal(3 * N) * 0.01).astype(np.float32)
    emb = (rng.standard_normal((layers, 3 * N)) * 0.01).astype(np.float32)
    dev = lambda x: torch.from_numpy(x).to(_gpu.DEV)  # noqa: E731
    for layer in (0, 5):
        got = tt.adaln_single(dev(t), dev(w1), dev(b1), dev(w2), dev(b2), dev(emb), layer)
        torch.cuda.synchronize()
        want = oracle.adaln_single(t, w1, b1, w2, b2, emb, layer)
        for g, w in zip(got, want):
            # fp32 dot products of length F and Dh against fp64
            assert np.abs(g.cpu().numpy() - w).max() <= 1e-5
