"""GPU parity of tt_kv_append: appending a committed block to every layer's context.

Byte work: caches, lengths and the overflow count must equal the oracle's exactly,
including every cache row the append must not touch.
"""
import numpy as np
import pytest
import torch

import oracle
from block_mask_diffusion_tt_b300 import synth, tt
import _gpu

pytestmark = pytest.mark.gpu


def _bits(rng, shape):
    return synth.bf16_bits(rng.standard_normal(shape).astype(np.float32))


def _to_np(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _case(seed, B, S, Hkv, d, Lmax, lens, layers):
    rng = np.random.default_rng(seed)
    kc = [_bits(rng, (B, Hkv, Lmax, d)) for _ in range(layers)]
    vc = [_bits(rng, (B, Hkv, Lmax, d)) for _ in range(layers)]
    kb = [_bits(rng, (B, S, Hkv, d)) for _ in range(layers)]
    vb = [_bits(rng, (B, S, Hkv, d)) for _ in range(layers)]
    return kc, vc, np.asarray(lens, np.int32), kb, vb


def _run_and_compare(kc, vc, lens, kb, vb, active=None, views=None):
    dk = [_gpu.bf16_dev(x) for x in kc] if views is None else views[0]
    dv = [_gpu.bf16_dev(x) for x in vc] if views is None else views[1]
    dl = torch.from_numpy(lens.copy()).to(_gpu.DEV)
    da = None if active is None else torch.from_numpy(active).to(_gpu.DEV)
    ovf = torch.zeros((1,), dtype=torch.int32, device=_gpu.DEV)
    tt.kv_append(dk, dv, dl, [_gpu.bf16_dev(x) for x in kb], [_gpu.bf16_dev(x) for x in vb],
                 active=da, overflow=ovf)
    torch.cuda.synchronize()
    ref = oracle.kv_append(kc, vc, lens, kb, vb, active=active)
    for layer in range(len(kc)):
        assert np.array_equal(_to_np(dk[layer]), ref["k_ctx"][layer]), f"k layer {layer}"
        assert np.array_equal(_to_np(dv[layer]), ref["v_ctx"][layer]), f"v layer {layer}"
    assert dl.cpu().numpy().tolist() == ref["ctx_lens"].tolist()
    assert int(ovf.item()) == ref["overflow"]
    return ref


def test_append_matches_oracle_with_edges():
    # empty prefix, mid, exact fit (84 + 16 = 100), one past (85), at the end (99),
    # an invalid negative length and an inactive sequence
    kc, vc, lens, kb, vb = _case(1, 7, 16, 2, 128, 100, [0, 50, 84, 85, 99, -3, 30], 3)
    active = np.array([1, 1, 1, 1, 1, 1, 0], np.uint8)
    ref = _run_and_compare(kc, vc, lens, kb, vb, active=active)
    assert ref["overflow"] == 3


@pytest.mark.parametrize("S,Hkv,d,layers", [(1, 1, 64, 1), (16, 2, 64, 6), (64, 4, 128, 2),
                                            (7, 3, 128, 16)])
def test_append_shapes(S, Hkv, d, layers):
    rng = np.random.default_rng(S + d)
    B, Lmax = 4, 3 * S + 5
    lens = rng.integers(0, 2 * S, size=B).astype(np.int32)
    kc, vc, lens, kb, vb = _case(S * 7 + Hkv, B, S, Hkv, d, Lmax, lens, layers)
    _run_and_compare(kc, vc, lens, kb, vb)


def test_append_into_strided_cache_views():
    """Caches that are views into larger buffers (a paged-style allocation)."""
    B, S, Hkv, d, Lmax = 3, 16, 2, 64, 40
    kc, vc, lens, kb, vb = _case(9, B, S, Hkv, d, Lmax, [0, 10, 24], 2)
    views = ([], [])
    for src, out in ((kc, views[0]), (vc, views[1])):
        for x in src:
            big = torch.zeros((B, Hkv, Lmax + 8, d + 64), dtype=torch.bfloat16, device=_gpu.DEV)
            v = big[:, :, 4:4 + Lmax, 32:32 + d]
            v.copy_(_gpu.bf16_dev(x))
            out.append(v)
    _run_and_compare(kc, vc, lens, kb, vb, views=views)


def test_two_blocks_of_generation():
    """Block 1 attends to the prefix; once it is committed its K/V are appended; block 2
    attends to the longer prefix.  Both attention calls against the oracle."""
    B, S, Hq, Hkv, d, Lmax = 2, 16, 8, 2, 128, 256
    shape = synth.AttnShape(B, S, Hq, Hkv, d, Lmax, lens=[100, 37])
    inp1 = synth.attn_inputs(shape, seed=40)
    _gpu.check_attn(inp1, what="block 1")
    dev = _gpu.attn_dev(inp1)
    lens = dev["ctx_lens"]
    tt.kv_append([dev["k_ctx"]], [dev["v_ctx"]], lens, [dev["k_blk"]], [dev["v_blk"]])
    torch.cuda.synchronize()
    grown = oracle.kv_append([inp1["k_ctx"]], [inp1["v_ctx"]], inp1["ctx_lens"], [inp1["k_blk"]],
                             [inp1["v_blk"]])
    assert lens.cpu().numpy().tolist() == [116, 53]
    inp2 = synth.attn_inputs(shape, seed=41)
    inp2.update(k_ctx=grown["k_ctx"][0], v_ctx=grown["v_ctx"][0], ctx_lens=grown["ctx_lens"])
    assert np.array_equal(_to_np(dev["k_ctx"]), inp2["k_ctx"])
    _gpu.check_attn(inp2, what="block 2 over the appended prefix")
