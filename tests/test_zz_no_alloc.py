"""tt_block_attn_noalloc: block attention for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc -- their device memory belongs to another
allocator's pool, or they run a loop that must not risk the device-wide
synchronisation an allocation can cause -- so they cannot provide the workspace
tt_block_attn asks for.  This entry point takes no workspace and allocates
nothing: its scratch is a fixed array inside libtt.  The test calls it through
the C ABI twice in a row (the second call reuses the scratch the first left
behind) and checks each output against the workspace entry point's, and against
the fp64 oracle, within the attention tolerances the other GPU tests use.  It runs
last so that a failure here cannot hide the results of the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from block_mask_diffusion_tt_b300 import synth, tt
import _gpu

pytestmark = pytest.mark.gpu


def _noalloc_raw(d, out, lse):
    """Direct C-ABI call of tt_block_attn_noalloc on device tensors."""
    lib = tt.load()
    fn = lib.tt_block_attn_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(tt.AttnDesc)] + [ctypes.c_void_p] * 9
    desc = tt.attn_desc(d["q"], d["k_ctx"], d["v_ctx"], d["k_blk"], d["v_blk"], out)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fn(ctypes.byref(desc), d["q"].data_ptr(), d["k_ctx"].data_ptr(),
              d["v_ctx"].data_ptr(), d["ctx_lens"].data_ptr(), d["k_blk"].data_ptr(),
              d["v_blk"].data_ptr(), out.data_ptr(), lse.data_ptr(), stream)


_RNG = np.random.default_rng(120)


@pytest.mark.parametrize("shape", [
    synth.AttnShape(4, 16, 32, 2, 128, 3000, lens=[3000, 17, 1500, 0]),
    synth.AttnShape(1, 16, 16, 1, 128, 40000, lens=[40000]),  # one pair over every SM
    synth.AttnShape(3, 16, 8, 2, 64, 700, lens=[700, 64, 300]),
    # 240 pairs at d=128: the scratch then holds fewer partial slots than the device has
    # SMs, so the prefix is split over a reduced number of CTAs
    synth.AttnShape(120, 16, 32, 2, 128, 300,
                    lens=[int(x) for x in _RNG.integers(0, 301, size=120)]),
], ids=["ragged", "long-single", "d64", "240-pairs"])
def test_noalloc_matches_workspace_entry_point_twice(shape):
    for call, seed in enumerate((21, 22)):
        inp = synth.attn_inputs(shape, seed=seed)
        d = _gpu.attn_dev(inp)
        B, S, Hq, D = inp["q"].shape
        ref_lse = torch.empty((B, Hq, S), dtype=torch.float32, device=_gpu.DEV)
        ref = tt.block_attn(d["q"], d["k_ctx"], d["v_ctx"], d["ctx_lens"], d["k_blk"], d["v_blk"],
                            lse=ref_lse)
        out = torch.full((B, S, Hq, D), float("nan"), dtype=torch.bfloat16, device=_gpu.DEV)
        lse = torch.full((B, Hq, S), float("nan"), dtype=torch.float32, device=_gpu.DEV)
        status = _noalloc_raw(d, out, lse)
        assert status == tt.TT_OK, tt.last_error()
        torch.cuda.synchronize()
        got = out.float().cpu().numpy().astype(np.float64)
        want = ref.float().cpu().numpy().astype(np.float64)
        _gpu.assert_attn_close(got, want, lse.cpu().numpy(), ref_lse.cpu().numpy(),
                               f"noalloc call {call + 1}")
        exact, exact_lse = oracle.block_attn(inp["q"], inp["k_ctx"], inp["v_ctx"],
                                             inp["ctx_lens"], inp["k_blk"], inp["v_blk"])
        _gpu.assert_attn_close(got, exact, lse.cpu().numpy(), exact_lse,
                               f"noalloc call {call + 1} against the oracle")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    B, S, Hq, Hkv, D = 126, 16, 32, 2, 128  # 252 pairs: more than the fixed scratch holds
    q = torch.zeros((B, S, Hq, D), dtype=torch.bfloat16, device=_gpu.DEV)
    kv = torch.zeros((B, Hkv, 8, D), dtype=torch.bfloat16, device=_gpu.DEV)
    blk = torch.zeros((B, S, Hkv, D), dtype=torch.bfloat16, device=_gpu.DEV)
    lens = torch.zeros((B,), dtype=torch.int32, device=_gpu.DEV)
    d = dict(q=q, k_ctx=kv, v_ctx=kv, k_blk=blk, v_blk=blk, ctx_lens=lens)
    out = torch.zeros_like(q)
    lse = torch.zeros((B, Hq, S), dtype=torch.float32, device=_gpu.DEV)
    assert _noalloc_raw(d, out, lse) == tt.TT_ERR_UNSUPPORTED
    assert "static scratch" in tt.last_error()
    assert (out == 0).all()  # nothing was launched
