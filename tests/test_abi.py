"""libtt loads, exports every entry point include/tt.h declares, and validates on the host.

No test here launches GPU work: every call below fails validation (or only
formats a status) before the library touches the CUDA runtime.
"""
import ctypes
import os
import re

import pytest

from block_mask_diffusion_tt_b300 import tt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(tt_\w+)\s*\(", text, flags=re.M):
            if not text[m.start():m.end()].lstrip().startswith("typedef"):
                names.append(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    return tt.load()


def test_header_declares_the_three_operations():
    names = header_functions()
    for n in ("tt_block_attn", "tt_confidence_unmask", "tt_denoise_block_loop"):
        assert n in names
    assert len(names) == len(set(names))


def test_every_declared_symbol_is_exported(lib):
    for n in header_functions():
        assert hasattr(lib, n), n
    assert sorted(header_functions()) == sorted(tt.exported_symbols())


def test_status_strings_and_version(lib):
    assert tt.status_string(tt.TT_OK) == "TT_OK"
    assert tt.status_string(tt.TT_ERR_TIMEOUT) == "TT_ERR_TIMEOUT"
    assert lib.tt_abi_version() == 1000


def _unmask_call(lib, desc):
    return lib.tt_confidence_unmask(ctypes.byref(desc) if desc is not None else None, None, None,
                                    None, None, None, None, 0, None, 0, None)


@pytest.mark.parametrize("kw,status", [
    (dict(S=0), tt.TT_ERR_INVALID_ARG), (dict(S=65), tt.TT_ERR_UNSUPPORTED),
    (dict(V=0), tt.TT_ERR_INVALID_ARG), (dict(B=-1), tt.TT_ERR_INVALID_ARG),
    (dict(temperature=0.0), tt.TT_ERR_INVALID_ARG), (dict(temperature=-1.0), tt.TT_ERR_INVALID_ARG),
    (dict(temperature=float("inf")), tt.TT_ERR_INVALID_ARG),
    (dict(threshold=float("nan")), tt.TT_ERR_INVALID_ARG),
    (dict(dtype=7), tt.TT_ERR_INVALID_ARG),
])
def test_unmask_rejects_bad_desc(lib, kw, status):
    base = dict(B=2, S=16, V=1024, dtype=tt.TT_BF16, temperature=0.1, threshold=0.8)
    base.update(kw)
    desc = tt.unmask_desc(base["B"], base["S"], base["V"], base["dtype"], base["temperature"],
                          base["threshold"], 3)
    assert _unmask_call(lib, desc) == status
    assert tt.last_error() != ""
    assert tt.confidence_unmask_workspace_size(desc) == 0


def test_unmask_rejects_null_desc_and_pointers(lib):
    assert _unmask_call(lib, None) == tt.TT_ERR_INVALID_ARG
    desc = tt.unmask_desc(2, 16, 1024, tt.TT_BF16, 0.1, 0.8, 3)
    assert _unmask_call(lib, desc) == tt.TT_ERR_INVALID_ARG  # null logits
    desc.logits_row_stride = 100  # < V
    assert _unmask_call(lib, desc) == tt.TT_ERR_INVALID_ARG


def test_unmask_workspace_size_is_host_only(lib):
    desc = tt.unmask_desc(8, 16, 131072, tt.TT_BF16, 0.1, 0.8, 3)
    n = tt.confidence_unmask_workspace_size(desc)
    assert n > 0 and n % 256 == 0
    assert tt.denoise_block_loop_workspace_size(desc) > n


def _attn_desc(**kw):
    p = dict(B=2, S=16, Hq=32, Hkv=2, d=128, Lmax=4096)
    p.update(kw)
    B, S, Hq, Hkv, d, L = (p[k] for k in ("B", "S", "Hq", "Hkv", "d", "Lmax"))
    desc = tt.AttnDesc(B=B, S=S, Hq=Hq, Hkv=Hkv, d=d, Lmax=L, scale=0.0)
    desc.q_strides = tt._i64x4(S * Hq * d, Hq * d, d, 1)
    desc.kctx_strides = tt._i64x4(Hkv * L * d, L * d, d, 1)
    desc.vctx_strides = tt._i64x4(Hkv * L * d, L * d, d, 1)
    desc.kblk_strides = tt._i64x4(S * Hkv * d, Hkv * d, d, 1)
    desc.vblk_strides = tt._i64x4(S * Hkv * d, Hkv * d, d, 1)
    desc.o_strides = tt._i64x4(S * Hq * d, Hq * d, d, 1)
    for k, v in p.items():
        if k.endswith("_strides"):
            setattr(desc, k, tt._i64x4(*v))
    return desc


def _attn_call(lib, desc):
    return lib.tt_block_attn(ctypes.byref(desc) if desc is not None else None, None, None, None,
                             None, None, None, None, None, None, 0, None)


@pytest.mark.parametrize("kw,status", [
    (dict(Hq=33), tt.TT_ERR_INVALID_ARG), (dict(d=96), tt.TT_ERR_UNSUPPORTED),
    (dict(S=0), tt.TT_ERR_INVALID_ARG), (dict(S=65), tt.TT_ERR_UNSUPPORTED),
    (dict(Lmax=-1), tt.TT_ERR_INVALID_ARG), (dict(B=-3), tt.TT_ERR_INVALID_ARG),
    (dict(q_strides=(16 * 32 * 128, 32 * 128, 128, 2)), tt.TT_ERR_UNSUPPORTED),
    (dict(kctx_strides=(2 * 4096 * 128, 4096 * 128, 132, 1)), tt.TT_ERR_UNSUPPORTED),
    (dict(B=4096), tt.TT_ERR_UNSUPPORTED),
])
def test_attn_rejects_bad_desc(lib, kw, status):
    assert _attn_call(lib, _attn_desc(**kw)) == status
    assert tt.block_attn_workspace_size(_attn_desc(**kw)) == 0


def test_attn_rejects_null_desc(lib):
    assert _attn_call(lib, None) == tt.TT_ERR_INVALID_ARG


def test_loop_rejects_bad_arguments(lib):
    desc = tt.unmask_desc(2, 16, 1024, tt.TT_F32, 0.1, 0.8, 3)
    steps = tt._i32(-1)
    call = lambda spb, start, prod: lib.tt_denoise_block_loop(  # noqa: E731
        ctypes.byref(desc), spb, start, 0, prod, None, None, None, None, None, None, None, 0, None,
        1000, ctypes.byref(steps))
    prod = ctypes.cast(lib.tt_synth_logits_producer, ctypes.c_void_p)
    assert call(0, 0, prod) == tt.TT_ERR_INVALID_ARG
    assert steps.value == 0
    assert call(16, 17, prod) == tt.TT_ERR_INVALID_ARG
    assert call(16, 0, None) == tt.TT_ERR_INVALID_ARG
    assert call(16, 0, prod) == tt.TT_ERR_INVALID_ARG  # null buffers


def test_synth_rejects_bad_arguments(lib):
    assert lib.tt_synth_logits(0, 0, 1, 16, 1024, 5, 2.0, 0, None, None) == tt.TT_ERR_INVALID_ARG
    assert lib.tt_synth_logits(0, -1, 1, 16, 1024, 1, 2.0, 0, None, None) == tt.TT_ERR_INVALID_ARG
    assert lib.tt_synth_logits(0, 0, 1, 16, 1024, 1, -2.0, 0, None, None) == tt.TT_ERR_INVALID_ARG
    assert lib.tt_synth_logits(0, 0, 1, 16, 1024, 1, 2.0, 0, None, None) == tt.TT_ERR_INVALID_ARG


def _kv_desc(**kw):
    base = dict(B=2, S=16, Hkv=2, d=128, Lmax=64, n_layers=2)
    base.update(kw)
    desc = tt.KvDesc(**base)
    desc.ctx_strides = tt._i64x4(2 * 64 * 128, 64 * 128, 128, 1)
    desc.blk_strides = tt._i64x4(16 * 2 * 128, 2 * 128, 128, 1)
    return desc


def _kv_call(lib, desc, ptr=None, n=2):
    arr = (ctypes.c_void_p * max(n, 1))(*([ptr] * max(n, 1)))
    lens = ctypes.c_void_p(ptr) if ptr else None
    return lib.tt_kv_append(ctypes.byref(desc) if desc is not None else None, arr, arr, lens, arr,
                            arr, None, None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(S=0), tt.TT_ERR_INVALID_ARG), (dict(Hkv=0), tt.TT_ERR_INVALID_ARG),
    (dict(B=-1), tt.TT_ERR_INVALID_ARG), (dict(Lmax=-1), tt.TT_ERR_INVALID_ARG),
    (dict(n_layers=0), tt.TT_ERR_INVALID_ARG), (dict(n_layers=17), tt.TT_ERR_INVALID_ARG),
    (dict(d=12), tt.TT_ERR_UNSUPPORTED), (dict(d=1024), tt.TT_ERR_UNSUPPORTED),
])
def test_kv_append_rejects_bad_desc(lib, kw, status):
    assert _kv_call(lib, _kv_desc(**kw)) == status


def test_kv_append_rejects_bad_strides_and_pointers(lib):
    d = _kv_desc()
    d.ctx_strides = tt._i64x4(2 * 64 * 128, 64 * 128, 128, 2)
    assert _kv_call(lib, d) == tt.TT_ERR_UNSUPPORTED  # innermost stride must be 1
    d = _kv_desc()
    d.blk_strides = tt._i64x4(16 * 2 * 128, 2 * 128, 100, 1)
    assert _kv_call(lib, d) == tt.TT_ERR_UNSUPPORTED  # not a multiple of 8 elements
    assert _kv_call(lib, None) == tt.TT_ERR_INVALID_ARG
    assert _kv_call(lib, _kv_desc()) == tt.TT_ERR_INVALID_ARG  # null pointers
    assert _kv_call(lib, _kv_desc(), ptr=0x100008) == tt.TT_ERR_INVALID_ARG  # not 16-byte aligned
    assert _kv_call(lib, _kv_desc(B=0)) == tt.TT_OK  # nothing to do: no launch


def test_state_seed_rejects_bad_desc(lib):
    desc = tt.StateDesc(B=2, n_layers=0, n_parts=1)
    assert lib.tt_mamba_state_seed(ctypes.byref(desc), None, None, None, None) == tt.TT_ERR_INVALID_ARG
    desc = tt.StateDesc(B=2, n_layers=1, n_parts=5)
    assert lib.tt_mamba_state_seed(ctypes.byref(desc), None, None, None, None) == tt.TT_ERR_INVALID_ARG
    desc = tt.StateDesc(B=2, n_layers=1, n_parts=1)
    desc.bytes[0] = 24  # not a multiple of 16
    desc.src_stride[0] = desc.dst_stride[0] = 32
    arr = (ctypes.c_void_p * 1)(16)
    assert lib.tt_mamba_state_seed(ctypes.byref(desc), arr, arr, None, None) == tt.TT_ERR_UNSUPPORTED
    assert "multiple of 16" in tt.last_error()


def test_generate_rejects_bad_params(lib):
    desc = tt.unmask_desc(2, 16, 100, tt.TT_BF16, 0.1, 0.8, 3)
    kv = tt.KvDesc(B=2, S=16, Hkv=2, d=64, Lmax=64, n_layers=1)
    gp = tt.GenerateParams(max_new_tokens=0, eos_token_id=-1, steps_per_block=16, timeout_ms=0)
    args = [None] * 17
    st = lib.tt_generate_blocks(ctypes.byref(desc), ctypes.byref(kv), ctypes.byref(gp), *args[:15],
                                None, 0, None, None)
    assert st == tt.TT_ERR_INVALID_ARG
    gp.max_new_tokens = 32
    kv.S = 8  # block size differs from the unmask desc
    st = lib.tt_generate_blocks(ctypes.byref(desc), ctypes.byref(kv), ctypes.byref(gp), *args[:15],
                                None, 0, None, None)
    assert st == tt.TT_ERR_INVALID_ARG and "B/S" in tt.last_error()
