"""The fp64 oracle against closed forms, invariants, library special cases and worked examples."""
import numpy as np
import pytest

import oracle
import _pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("check", _pins.ALL_CHECKS, ids=lambda f: f.__name__[len("check_"):])
def test_pin(check, lib):
    check(lib)


def test_ambiguity_flag_marks_only_fragile_decisions(lib):
    """The oracle flags decisions a 1e-5 relative error in a confidence could flip."""
    a = np.float32(np.log(4.0))  # conf = 1/(1+e^-a) = 0.8 up to fp32 rounding of a
    logits = np.array([[[a, 0.0], [0.0, 0.0]]], np.float32)
    r = oracle.confidence_unmask(logits, "f32", 1.0, 0.8, 3, np.full((1, 2), 3, np.int32),
                                 np.ones((1, 2), np.uint8), lib=lib)
    assert r["ambiguous"].tolist() == [[1, 0]]
    # confidences that are 1.0f on any fp32 evaluation tie exactly: not ambiguous
    spiky = np.zeros((1, 3, 50), np.float32)
    spiky[0, :, 7] = 30.0
    r = oracle.confidence_unmask(spiky, "f32", 0.1, 1.5, 3, np.full((1, 3), 3, np.int32),
                                 np.ones((1, 3), np.uint8), lib=lib)
    assert not r["ambiguous"].any() and r["committed_now"].tolist() == [[1, 0, 0]]
    # a fallback between two near-equal confidences below one is ambiguous
    near = np.zeros((1, 2, 4), np.float32)
    near[0, 0, 0] = 1.0
    near[0, 1, 0] = np.nextafter(np.float32(1.0), np.float32(2.0))
    r = oracle.confidence_unmask(near, "f32", 1.0, 0.99, 3, np.full((1, 2), 3, np.int32),
                                 np.ones((1, 2), np.uint8), lib=lib)
    assert r["ambiguous"].tolist() == [[1, 1]]


def _append_one_row_late(k_ctx, v_ctx, ctx_lens, k_blk, v_blk, active=None):
    lens = np.asarray(ctx_lens) + 1  # planted mistake: the block lands one row after the prefix
    r = oracle.kv_append(k_ctx, v_ctx, lens, k_blk, v_blk, active)
    r["ctx_lens"] = np.asarray(ctx_lens, np.int32) + k_blk[0].shape[1]
    return r


def _append_heads_and_rows_swapped(k_ctx, v_ctx, ctx_lens, k_blk, v_blk, active=None):
    # planted mistake: block [B,S,Hkv,d] read as if it were [B,Hkv,S,d]
    sw = lambda t: np.ascontiguousarray(t.reshape(t.shape[0], t.shape[2], t.shape[1], t.shape[3])  # noqa: E731
                                        .transpose(0, 2, 1, 3))
    return oracle.kv_append(k_ctx, v_ctx, ctx_lens, [sw(x) for x in k_blk],
                            [sw(x) for x in v_blk], active)


@pytest.mark.parametrize("mutant", [_append_one_row_late, _append_heads_and_rows_swapped])
def test_kv_append_pin_catches_planted_mistakes(lib, mutant):
    with pytest.raises(AssertionError):
        _pins.kv_append_then_attend(lib, append_fn=mutant)
