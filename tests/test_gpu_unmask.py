"""GPU parity of tt_confidence_unmask against the fp64 oracle (bit-exact ids and commits)."""
import ctypes

import numpy as np
import pytest
import torch

from block_mask_diffusion_tt_b300 import synth, tt
import _gpu

pytestmark = pytest.mark.gpu


def test_tiny_config_step0():
    w = synth.workloads()["tiny"]
    logits = synth.counter_logits(w.seed, 0, w.attn.B, w.attn.S, w.V, w.sigma, w.spike_p, "f32")
    _gpu.check_unmask(logits, "f32", w.temperature, w.threshold, w.mask_token_id)


@pytest.mark.parametrize("name", ["default", "ragged16k", "long"])
def test_full_size_configs(name):
    w = synth.workloads()[name]
    logits = synth.counter_logits(w.seed, 0, w.attn.B, w.attn.S, w.V, w.sigma, w.spike_p, "bf16")
    ref, _ = _gpu.check_unmask(logits, "bf16", w.temperature, w.threshold, w.mask_token_id)
    assert ref["committed_now"].sum() > 0


@pytest.mark.parametrize("gamma", [0.0, 0.5, 0.95, 1.5])
@pytest.mark.parametrize("V", [1, 7, 1000, 4099, 20000, 131072])
def test_vocab_sizes_and_thresholds(V, gamma):
    # ragged V exercises unaligned rows, scalar heads/tails and several chunks
    logits = synth.counter_logits(5, 1, 3, 16, V, 1.0, 0.4, "bf16")
    _gpu.check_unmask(logits, "bf16", 0.1, gamma)


@pytest.mark.parametrize("V", [3, 1023, 65537])
def test_fp32_logits(V):
    logits = synth.counter_logits(6, 2, 2, 8, V, 3.0, 0.3, "f32")
    _gpu.check_unmask(logits, "f32", 0.1, 0.8)


def test_partial_mask_state_and_remask():
    rng = np.random.default_rng(0)
    B, S, V = 4, 16, 5000
    logits = synth.counter_logits(7, 0, B, S, V, 0.5, 0.2, "bf16")
    masked = (rng.random((B, S)) < 0.6).astype(np.uint8)
    masked[2] = 0  # a finished sequence
    tokens = np.where(masked == 1, 99, rng.integers(0, V, (B, S))).astype(np.int32)
    ref, got = _gpu.check_unmask(logits, "bf16", 0.1, 0.9, tokens=tokens, masked=masked)
    assert got["remaining"][2] == 0 and not got["committed_now"][2].any()


def test_force_commit_all():
    logits = synth.counter_logits(8, 0, 2, 32, 3000, 0.5, 0.0, "bf16")
    masked = np.ones((2, 32), np.uint8)
    masked[0, ::3] = 0
    _gpu.check_unmask(logits, "bf16", 0.1, 0.99, masked=masked, force=True)


def test_planted_ties_pick_lowest_index():
    B, S, V = 2, 8, 40000
    logits = synth.counter_logits(9, 0, B, S, V, 1.0, 0.0, "f32")
    for r, idx in enumerate([[5, 39999], [17000, 17001, 3], [100, 20000, 30000], [0, 1]]):
        logits.reshape(B * S, V)[r, idx] = 50.0
    ref, got = _gpu.check_unmask(logits, "f32", 0.1, 0.0)
    flat = got["tokens"].reshape(-1)
    assert flat[0] == 5 and flat[1] == 3 and flat[2] == 100 and flat[3] == 0


def test_fallback_tie_lowest_position():
    B, S, V = 1, 8, 64
    logits = np.zeros((B, S, V), np.float32)
    logits[0, :, :] = np.random.default_rng(1).standard_normal((S, V)).astype(np.float32) * 0.01
    logits[0, 5] = logits[0, 2]
    logits[0, 2, 10] = logits[0, 5, 10] = 0.3
    ref, got = _gpu.check_unmask(logits, "f32", 0.1, 0.9, allow_ambiguous=True)
    assert got["committed_now"][0].tolist() == [0, 0, 1, 0, 0, 0, 0, 0]
    assert got["tokens"][0, 2] == 10


def test_row_stride_padding():
    B, S, V, pad = 2, 16, 1000, 24
    full = synth.counter_logits(10, 0, B, S, V + pad, 1.0, 0.5, "bf16")
    t = _gpu.bf16_dev(full)[:, :, :V]
    logits = full[:, :, :V].copy()
    ref_tok = np.full((B, S), 3, np.int32)
    tok = torch.from_numpy(ref_tok.copy()).to(_gpu.DEV)
    msk = torch.ones((B, S), dtype=torch.uint8, device=_gpu.DEV)
    r = tt.confidence_unmask(t, tok, msk, 0.1, 0.8, 3)
    torch.cuda.synchronize()
    import oracle
    o = oracle.confidence_unmask(logits, "bf16", 0.1, 0.8, 3, ref_tok, np.ones((B, S), np.uint8))
    assert np.array_equal(r["tokens"].cpu().numpy(), o["tokens"])
    assert np.array_equal(r["committed_now"].cpu().numpy(), o["committed_now"])


def test_repeated_calls_reuse_workspace():
    """Many calls on one workspace stay exact (the kernels keep no state between calls
    beyond the error word, which stays 0)."""
    B, S, V = 3, 16, 50000
    desc = tt.unmask_desc(B, S, V, tt.TT_BF16, 0.1, 0.8, 3)
    ws = tt.Workspace(tt.confidence_unmask_workspace_size(desc))
    import oracle
    for step in range(4):
        logits = synth.counter_logits(11, step, B, S, V, 1.0, 0.3, "bf16")
        tok = np.full((B, S), 3, np.int32)
        msk = np.ones((B, S), np.uint8)
        o = oracle.confidence_unmask(logits, "bf16", 0.1, 0.8, 3, tok, msk)
        tok_d = torch.from_numpy(tok).to(_gpu.DEV)
        msk_d = torch.from_numpy(msk).to(_gpu.DEV)
        tt.confidence_unmask(_gpu.bf16_dev(logits), tok_d, msk_d, 0.1, 0.8, 3, workspace=ws)
        torch.cuda.synchronize()
        assert np.array_equal(tok_d.cpu().numpy(), o["tokens"])
    flag = ctypes.c_int32(-1)
    tt.check(tt.load().tt_confidence_unmask_error(ws.ptr, ctypes.byref(flag), None))
    assert flag.value == 0


def test_empty_batch_is_noop():
    tok = torch.zeros((0, 16), dtype=torch.int32, device=_gpu.DEV)
    msk = torch.zeros((0, 16), dtype=torch.uint8, device=_gpu.DEV)
    logits = torch.zeros((0, 16, 100), dtype=torch.bfloat16, device=_gpu.DEV)
    desc = tt.unmask_desc(0, 16, 100, tt.TT_BF16, 0.1, 0.8, 3)
    assert tt.confidence_unmask_workspace_size(desc) >= 0
    ws = tt.Workspace(256)
    tt.confidence_unmask(logits, tok, msk, 0.1, 0.8, 3, workspace=ws)


@pytest.mark.parametrize("B,S,V,dtype", [(40, 16, 4099, "bf16"), (40, 16, 20000, "f32"),
                                         (8, 16, 131072, "bf16"), (40, 16, 70001, "bf16"),
                                         (2, 16, 131072, "bf16"), (1, 16, 131072, "bf16")])
def test_grid_plans_and_unaligned_rows(B, S, V, dtype):
    """Units of 32 KB, and (on 148 SMs, three CTAs each) the 16 KB and 8 KB units of
    batches with fewer 32 KB units than CTAs (32 and 16 rows of 131072), with rows that
    start off a 16-byte boundary (odd V)."""
    logits = synth.counter_logits(12, 0, B, S, V, 1.0, 0.3, dtype)
    _gpu.check_unmask(logits, dtype, 0.1, 0.8)


def test_rows_with_negative_infinity():
    """-inf logits weigh nothing; a whole vocabulary chunk of -inf adds nothing."""
    B, S, V = 40, 16, 131072
    logits = synth.counter_logits(13, 0, B, S, V, 1.0, 0.3, "f32")
    flat = logits.reshape(B * S, V)
    flat[0, :70000] = -np.inf   # two whole chunks and part of a third
    flat[1, 1::2] = -np.inf
    flat[2, :V - 1] = -np.inf   # one finite logit
    _gpu.check_unmask(logits, "f32", 0.1, 0.8)


def test_rows_not_masked_cost_no_wait():
    """A step where most rows are already committed: their units are posted without
    data.  The call must finish promptly and leave the error word at 0 (every wait of
    the kernel is bounded at 2 s and a wait that runs out sets the word)."""
    import time
    B, S, V = 16, 16, 131072
    logits = synth.counter_logits(14, 0, B, S, V, 2.0, 0.6, "bf16")
    rng = np.random.default_rng(14)
    masked = (rng.random((B, S)) < 0.2).astype(np.uint8)
    tokens = np.where(masked == 1, 3, 7).astype(np.int32)
    desc = tt.unmask_desc(B, S, V, tt.TT_BF16, 0.1, 0.8, 3)
    ws = tt.Workspace(tt.confidence_unmask_workspace_size(desc))
    lg = _gpu.bf16_dev(logits)
    for rep in range(3):
        tok_d = torch.from_numpy(tokens.copy()).to(_gpu.DEV)
        msk_d = torch.from_numpy(masked.copy()).to(_gpu.DEV)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        tt.confidence_unmask(lg, tok_d, msk_d, 0.1, 0.8, 3, workspace=ws)
        torch.cuda.synchronize()
        assert time.perf_counter() - t0 < 0.5
    flag = ctypes.c_int32(-1)
    tt.check(tt.load().tt_confidence_unmask_error(ws.ptr, ctypes.byref(flag), None))
    assert flag.value == 0
    _gpu.check_unmask(logits, "bf16", 0.1, 0.8, tokens=tokens, masked=masked)
