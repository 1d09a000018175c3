"""GPU parity of tt_generate_blocks (block-by-block generation) against the oracle.

Both sides use the same stand-ins: per-(block, step) counter-generated logits (the
device generator and its Python twin are bit-identical) for the denoiser forward,
and per-(block, layer) counter-generated K/V for the context tower.  Everything the
call produces is compared exactly: generated tokens, lengths, active flags, the
steps taken, the overflow count, context lengths and every row of every cache.
"""
import numpy as np
import pytest
import torch

import oracle
from block_mask_diffusion_tt_b300 import synth, tt
import _gpu

pytestmark = pytest.mark.gpu


def _kv_seed(kind, block, layer, layers):
    return (1000 if kind == "k" else 2000) + block * layers + layer


def _case(B, S, V, Hkv, d, layers, Lmax, lens, max_new, eos, gamma, steps=None, active=None,
          seed=7, sigma=1.0, p=0.3, T=0.1):
    steps = steps or S
    rng = np.random.default_rng(seed)
    kc = [synth.bf16_bits(rng.standard_normal((B, Hkv, Lmax, d)).astype(np.float32))
          for _ in range(layers)]
    vc = [synth.bf16_bits(rng.standard_normal((B, Hkv, Lmax, d)).astype(np.float32))
          for _ in range(layers)]
    lens = np.asarray(lens, np.int32)
    act = np.ones(B, np.uint8) if active is None else np.asarray(active, np.uint8)
    thr = synth.spike_threshold(p)

    # ---- oracle
    def logits_np(block, step):
        return synth.counter_logits(seed + block, step, B, S, V, sigma, p, "bf16")

    def kv_np(block, tokens):
        k = [synth.counter_logits(_kv_seed("k", block, l, layers), 0, B, S, Hkv * d, 1.0, 0.0,
                                  "bf16").reshape(B, S, Hkv, d) for l in range(layers)]
        v = [synth.counter_logits(_kv_seed("v", block, l, layers), 0, B, S, Hkv * d, 1.0, 0.0,
                                  "bf16").reshape(B, S, Hkv, d) for l in range(layers)]
        return k, v

    ref = oracle.generate_blocks(B, S, logits_np, kv_np, kc, vc, lens, "bf16", T, gamma, 3,
                                 steps, max_new, eos, active=act, out_fill=-1)
    assert ref["ambiguous"] == 0

    # ---- device
    dk = [_gpu.bf16_dev(x) for x in kc]
    dv = [_gpu.bf16_dev(x) for x in vc]
    kb = [torch.empty((B, S, Hkv, d), dtype=torch.bfloat16, device=_gpu.DEV) for _ in range(layers)]
    vb = [torch.empty((B, S, Hkv, d), dtype=torch.bfloat16, device=_gpu.DEV) for _ in range(layers)]
    dl = torch.from_numpy(lens.copy()).to(_gpu.DEV)
    out = torch.full((B, max_new), -1, dtype=torch.int32, device=_gpu.DEV)
    gen_len = torch.zeros((B,), dtype=torch.int32, device=_gpu.DEV)
    dact = torch.from_numpy(act.copy()).to(_gpu.DEV)
    steps_total = torch.zeros((B,), dtype=torch.int32, device=_gpu.DEV)
    ovf = torch.zeros((1,), dtype=torch.int32, device=_gpu.DEV)

    def logits_dev(block, step, buf):
        tt.synth_logits(seed + block, step, B, S, V, sigma, thr, tt.TT_BF16, out=buf)

    def kv_dev(block, tokens, active, k_blk, v_blk):
        for l in range(layers):
            tt.synth_logits(_kv_seed("k", block, l, layers), 0, B, S, Hkv * d, 1.0, 0, tt.TT_BF16,
                            out=k_blk[l].view(B, S, Hkv * d))
            tt.synth_logits(_kv_seed("v", block, l, layers), 0, B, S, Hkv * d, 1.0, 0, tt.TT_BF16,
                            out=v_blk[l].view(B, S, Hkv * d))

    n = tt.generate_blocks(logits_dev, kv_dev, V, tt.TT_BF16, T, gamma, 3, steps, max_new, eos,
                           dk, dv, dl, kb, vb, out, gen_len, dact, steps_total, ovf)
    torch.cuda.synchronize()
    assert n == ref["blocks_run"]
    assert np.array_equal(out.cpu().numpy(), ref["out_tokens"])
    live = act == 1
    assert np.array_equal(gen_len.cpu().numpy()[live], ref["gen_len"][live])
    assert np.array_equal(dact.cpu().numpy(), ref["active"])
    assert np.array_equal(steps_total.cpu().numpy(), ref["steps_total"])
    assert int(ovf.item()) == ref["overflow"]
    assert np.array_equal(dl.cpu().numpy(), ref["ctx_lens"])
    for l in range(layers):
        assert np.array_equal(dk[l].view(torch.int16).cpu().numpy().view(np.uint16), ref["k_ctx"][l])
        assert np.array_equal(dv[l].view(torch.int16).cpu().numpy().view(np.uint16), ref["v_ctx"][l])
    return ref


def test_natural_eos_small_vocabulary():
    """V = 64: EOS (id 5) is the argmax of some positions, so sequences stop at different
    blocks; lengths count up to the first EOS."""
    ref = _case(B=6, S=8, V=64, Hkv=2, d=64, layers=2, Lmax=128, lens=[0, 3, 17, 40, 8, 29],
                max_new=40, eos=5, gamma=0.8)
    assert len(set(ref["gen_len"].tolist())) > 1  # the case does exercise EOS stops


def test_capacity_inactive_and_partial_last_block():
    """max_new = 2S + 3 (the last block keeps 3 positions), one sequence inactive from
    the start, one whose cache fills up after its first appended block."""
    ref = _case(B=4, S=8, V=300, Hkv=1, d=64, layers=3, Lmax=30, lens=[0, 14, 5, 20],
                max_new=19, eos=-1, gamma=0.9, active=[1, 1, 0, 1])
    assert ref["overflow"] > 0


def test_wide_vocabulary_four_blocks():
    _case(B=8, S=16, V=4099, Hkv=2, d=128, layers=2, Lmax=256, lens=[0, 1, 63, 64, 65, 100, 150, 7],
          max_new=64, eos=11, gamma=0.8, p=0.6, sigma=2.0)


def test_one_commit_per_step_counts_steps():
    """gamma > 1: each block takes exactly S steps, so steps_total = S x blocks."""
    # no spikes, small sigma: the fallback choices between positions are clear in fp32
    ref = _case(B=3, S=4, V=128, Hkv=2, d=64, layers=1, Lmax=64, lens=[2, 0, 9], max_new=12,
                eos=-1, gamma=1.5, seed=9, sigma=0.5, p=0.0)
    assert ref["steps_total"].tolist() == [12, 12, 12]
