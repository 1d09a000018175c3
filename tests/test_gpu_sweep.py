"""GPU parity on the block-size and threshold sweep workload.

Sweep shape: B=16, L=8192, S in {4, 8, 16, 32, 64}, Hq=32, Hkv=2, d=128, V=131072,
steps_per_block = S, gamma in {0.5, 0.8, 0.95}, logits regenerated per step with a
spike probability growing linearly from 0.2 to 0.9 across the steps.

* Block loop: the whole batch runs on the GPU through tt_denoise_block_loop with the
  library's counter-based producer; the first sequences are replayed in the oracle
  (rows b*S+s of the first sequences are the same draws in a smaller batch) and
  compared bit for bit: tokens, is_masked, steps_used and committed_step.
* One unmask step over every row at S=4 and at S=64 (the kernel's largest block).
* Attention at S=4 and S=64 on the full sweep shape, sampled sequences in the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from block_mask_diffusion_tt_b300 import synth, tt
import _gpu

pytestmark = pytest.mark.gpu

W = synth.workloads()["sweep"]
S_VALUES = W.extra["S_values"]
GAMMAS = W.extra["gammas"]


def _state(B, S):
    return (torch.zeros((B, S), dtype=torch.int32, device=_gpu.DEV),
            torch.zeros((B, S), dtype=torch.uint8, device=_gpu.DEV),
            torch.zeros((B,), dtype=torch.int32, device=_gpu.DEV),
            torch.zeros((B, S), dtype=torch.int32, device=_gpu.DEV))


@pytest.mark.parametrize("gamma", GAMMAS)
@pytest.mark.parametrize("S", S_VALUES)
def test_sweep_loop_matches_oracle(S, gamma):
    B, V = W.attn.B, W.V
    ps = [synth.sweep_spike_p(k, S) for k in range(S)]
    tokens, masked, steps_used, cstep = _state(B, S)
    params = tt.synth_params(W.seed, B, S, V, tt.TT_BF16, W.sigma, _gpu.synth_thresholds(ps))
    n = tt.denoise_block_loop(B, S, V, tt.TT_BF16, W.temperature, gamma, W.mask_token_id, S,
                              tokens, masked, steps_used, cstep, synth=params)
    torch.cuda.synchronize()
    assert not masked.any(), "steps_per_block = S must finish every block"
    Bs = 2
    ref = oracle.block_loop(
        Bs, S, lambda k: synth.counter_logits(W.seed, k, Bs, S, V, W.sigma, ps[k], "bf16"),
        "bf16", W.temperature, gamma, W.mask_token_id, S)
    assert ref["ambiguous"] == 0
    got = {k: v.cpu().numpy()[:Bs] for k, v in
           dict(tokens=tokens, is_masked=masked, steps_used=steps_used,
                committed_step=cstep).items()}
    for k in ("tokens", "is_masked", "steps_used", "committed_step"):
        assert np.array_equal(got[k], ref[k]), k
    assert n >= int(ref["steps_used"].max())
    # every position was committed exactly once, at a step below S
    cs = cstep.cpu().numpy()
    assert (cs >= 0).all() and (cs < S).all()


@pytest.mark.parametrize("S", [4, 64])
def test_unmask_step_every_row(S):
    """One unmask step over all B*S rows at the sweep's smallest and largest block."""
    B, V = W.attn.B, W.V
    logits = synth.counter_logits(W.seed, 0, B, S, V, W.sigma, synth.sweep_spike_p(0, S), "bf16")
    for gamma in (0.5, 0.95):
        ref, got = _gpu.check_unmask(logits, "bf16", W.temperature, gamma, W.mask_token_id)
        assert got["committed_now"].sum(axis=1).min() >= 1  # at least one per sequence


def test_unmask_s64_partial_state_and_fallback():
    """S = 64 with most positions already committed and a threshold above 1: the
    per-sequence commit keeps its 64-entry state in shared memory; exactly one
    position commits per sequence."""
    B, S, V = 8, 64, 131072
    rng = np.random.default_rng(64)
    # no spikes: with spikes several rows reach confidences just below 1.0f, and the
    # fallback between them is too close to call in fp32 (the oracle flags it)
    logits = synth.counter_logits(3, 1, B, S, V, W.sigma, 0.0, "bf16")
    masked = (rng.random((B, S)) < 0.3).astype(np.uint8)
    masked[:, 63] = 1  # the last position of every sequence is masked
    masked[5] = 0
    tokens = np.where(masked == 1, 3, rng.integers(0, V, (B, S))).astype(np.int32)
    ref, got = _gpu.check_unmask(logits, "bf16", W.temperature, 1.5, tokens=tokens, masked=masked)
    n = got["committed_now"].sum(axis=1)
    assert (n[masked.any(axis=1)] == 1).all() and n[5] == 0


@pytest.mark.parametrize("S", [4, 64])
def test_sweep_attention_sampled(S):
    shape = synth.AttnShape(W.attn.B, S, W.attn.Hq, W.attn.Hkv, W.attn.d, W.attn.Lmax)
    inp = synth.attn_inputs(shape, seed=W.seed + S)
    out, lse = _gpu.run_attn(inp)
    for b in (0, 11):
        sub = {k: inp[k][b:b + 1] for k in ("q", "k_ctx", "v_ctx", "k_blk", "v_blk", "ctx_lens")}
        ref, ref_lse = oracle.block_attn(sub["q"], sub["k_ctx"], sub["v_ctx"], sub["ctx_lens"],
                                         sub["k_blk"], sub["v_blk"])
        _gpu.assert_attn_close(out[b:b + 1], ref, lse[b:b + 1], ref_lse, f"sweep S={S} b={b}")
