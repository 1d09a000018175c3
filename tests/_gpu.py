"""Helpers shared by the GPU parity tests: uploads and comparisons against the oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from block_mask_diffusion_tt_b300 import synth, tt

# Tolerances.  Attention outputs: max-abs 1.5e-2 and mean-abs 2e-3 against the
# fp64 oracle on the same bf16 inputs; log-sum-exp 1e-4 absolute; confidences
# 1e-5 relative; token ids and commit flags bit-exact.
ATTN_MAX_ABS = 1.5e-2
ATTN_MEAN_ABS = 2e-3
LSE_ABS = 1e-4
CONF_REL = 1e-5

DEV = "cuda:0"


def bf16_dev(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def logits_dev(logits: np.ndarray, dtype: str) -> torch.Tensor:
    if dtype == "f32":
        return torch.from_numpy(np.ascontiguousarray(logits, dtype=np.float32)).to(DEV)
    return bf16_dev(logits)


def attn_dev(inp: dict) -> dict:
    out = {k: bf16_dev(inp[k]) for k in ("q", "k_ctx", "v_ctx", "k_blk", "v_blk")}
    out["ctx_lens"] = torch.from_numpy(inp["ctx_lens"].astype(np.int32)).to(DEV)
    return out


def run_attn(inp: dict, scale: float = 0.0, with_lse: bool = True, workspace=None):
    d = attn_dev(inp)
    B, S, Hq, _ = inp["q"].shape
    lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device=DEV) if with_lse else None
    out = tt.block_attn(d["q"], d["k_ctx"], d["v_ctx"], d["ctx_lens"], d["k_blk"], d["v_blk"],
                        lse=lse, scale=scale, workspace=workspace)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), (
        lse.cpu().numpy().astype(np.float64) if with_lse else None)


def assert_attn_close(out, ref, lse=None, ref_lse=None, what=""):
    assert np.isfinite(out).all(), f"{what}: non-finite output"
    err = np.abs(out - ref)
    assert err.max() <= ATTN_MAX_ABS, f"{what}: max-abs {err.max():.3e}"
    assert err.mean() <= ATTN_MEAN_ABS, f"{what}: mean-abs {err.mean():.3e}"
    if lse is not None:
        e2 = np.abs(lse - ref_lse)
        assert e2.max() <= LSE_ABS, f"{what}: lse max-abs {e2.max():.3e}"
    return float(err.max()), float(err.mean())


def check_attn(inp: dict, scale: float = 0.0, what: str = ""):
    out, lse = run_attn(inp, scale)
    ref, ref_lse = oracle.block_attn(inp["q"], inp["k_ctx"], inp["v_ctx"], inp["ctx_lens"],
                                     inp["k_blk"], inp["v_blk"], scale=scale)
    return assert_attn_close(out, ref, lse, ref_lse, what)


def check_unmask(logits: np.ndarray, dtype: str, T: float, gamma: float, mask_id: int = 3,
                 tokens=None, masked=None, force: bool = False, allow_ambiguous: bool = False):
    """One unmask step on both sides; bit-exact ids/flags, conf within CONF_REL."""
    B, S, _ = logits.shape
    tokens = np.full((B, S), mask_id, np.int32) if tokens is None else np.asarray(tokens, np.int32)
    masked = np.ones((B, S), np.uint8) if masked is None else np.asarray(masked, np.uint8)
    ref = oracle.confidence_unmask(logits, dtype, T, gamma, mask_id, tokens, masked,
                                   force_commit_all=force)
    amb = ref["ambiguous"].astype(bool)
    if not allow_ambiguous:
        assert not amb.any(), "seeded case hits a near-threshold decision"
    tok_d = torch.from_numpy(tokens.copy()).to(DEV)
    msk_d = torch.from_numpy(masked.copy()).to(DEV)
    r = tt.confidence_unmask(logits_dev(logits, dtype), tok_d, msk_d, T, gamma, mask_id,
                             force_commit_all=force)
    torch.cuda.synchronize()
    got = {k: v.cpu().numpy() for k, v in r.items()}
    ok_seq = ~amb.any(axis=1)
    for k in ("tokens", "is_masked", "committed_now"):
        assert np.array_equal(got[k][ok_seq], ref[k][ok_seq]), k
    assert np.array_equal(got["remaining"][ok_seq], ref["remaining"][ok_seq])
    was = masked == 1
    c_ref, c_got = ref["conf"][was], got["conf"][was].astype(np.float64)
    rel = np.abs(c_got - c_ref) / c_ref
    assert rel.max(initial=0.0) <= CONF_REL, f"conf rel err {rel.max():.3e}"
    assert np.isnan(got["conf"][~was]).all()
    return ref, got


def synth_thresholds(p_list) -> list:
    return [synth.spike_threshold(p) for p in p_list]
