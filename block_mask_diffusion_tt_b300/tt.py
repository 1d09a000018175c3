"""Thin ctypes binding of libtt (include/tt.h) taking torch CUDA tensors.

Argument marshalling only: shapes and strides are read from the tensors, the
raw device pointers and the current CUDA stream are passed to the C ABI, and a
non-OK status raises ``TTError``.  Every step of the computation runs in the
library's CUDA kernels; there is no fallback path, and loading fails loudly if
libtt.so has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Callable, Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtt.so")

TT_OK, TT_ERR_INVALID_ARG, TT_ERR_UNSUPPORTED, TT_ERR_WORKSPACE = 0, 1, 2, 3
TT_ERR_CUDA, TT_ERR_TIMEOUT, TT_ERR_CALLBACK, TT_ERR_INTERNAL = 4, 5, 6, 7
TT_F32, TT_BF16 = 0, 1
SYNTH_MAX_STEPS = 256
KV_MAX_LAYERS = 16

_i32 = ctypes.c_int32
_p = ctypes.c_void_p
_sz = ctypes.c_size_t
_i64x4 = ctypes.c_int64 * 4


class TTError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


class AttnDesc(ctypes.Structure):
    _fields_ = [("B", _i32), ("S", _i32), ("Hq", _i32), ("Hkv", _i32), ("d", _i32),
                ("Lmax", _i32), ("scale", ctypes.c_float), ("q_strides", _i64x4),
                ("kctx_strides", _i64x4), ("vctx_strides", _i64x4), ("kblk_strides", _i64x4),
                ("vblk_strides", _i64x4), ("o_strides", _i64x4)]


TT_KEYS_ALL, TT_KEYS_PREFIX, TT_KEYS_BLOCK = 0, 1, 2


class AttnOpts(ctypes.Structure):
    _fields_ = [("keys", _i32), ("block_table", _p), ("max_pages", _i32), ("n_pages", _i32),
                ("q_scale", _p), ("q_shift", _p), ("o_gate", _p)]


class AdalnDesc(ctypes.Structure):
    _fields_ = [("B", _i32), ("F", _i32), ("Dh", _i32), ("N", _i32), ("layer", _i32),
                ("n_layers", _i32)]


class UnmaskDesc(ctypes.Structure):
    _fields_ = [("B", _i32), ("S", _i32), ("V", _i32), ("logits_dtype", ctypes.c_int),
                ("logits_row_stride", ctypes.c_int64), ("temperature", ctypes.c_float),
                ("threshold", ctypes.c_float), ("mask_token_id", _i32)]


class SynthParams(ctypes.Structure):
    _fields_ = [("seed", ctypes.c_uint64), ("B", _i32), ("S", _i32), ("V", _i32),
                ("dtype", ctypes.c_int), ("sigma", ctypes.c_float),
                ("spike_threshold", ctypes.c_uint64 * SYNTH_MAX_STEPS)]


class KvDesc(ctypes.Structure):
    _fields_ = [("B", _i32), ("S", _i32), ("Hkv", _i32), ("d", _i32), ("Lmax", _i32),
                ("n_layers", _i32), ("ctx_strides", _i64x4), ("blk_strides", _i64x4)]


LOGITS_FN = ctypes.CFUNCTYPE(ctypes.c_int, _p, _i32, _p, _p, _p, _p)
BLOCK_LOGITS_FN = ctypes.CFUNCTYPE(ctypes.c_int, _p, _i32, _i32, _p, _p, _p, _p)
BLOCK_KV_FN = ctypes.CFUNCTYPE(ctypes.c_int, _p, _i32, _p, _p, _p, _p, _p)


STATE_MAX_LAYERS, STATE_MAX_PARTS = 64, 4
_i64xP = ctypes.c_int64 * STATE_MAX_PARTS


class StateDesc(ctypes.Structure):
    _fields_ = [("B", _i32), ("n_layers", _i32), ("n_parts", _i32), ("bytes", _i64xP),
                ("src_stride", _i64xP), ("dst_stride", _i64xP)]


class GenerateParams(ctypes.Structure):
    _fields_ = [("max_new_tokens", _i32), ("eos_token_id", _i32), ("steps_per_block", _i32),
                ("timeout_ms", _i32)]

_lib = None


def load(path: str = LIB_PATH):
    """Loads libtt.so (raises if it is missing: build it with build.py)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run `python -m block_mask_diffusion_tt_b300.build`")
    lib = ctypes.CDLL(path)
    sig = {
        "tt_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "tt_last_error": (ctypes.c_char_p, []),
        "tt_abi_version": (_i32, []),
        "tt_workspace_zero": (ctypes.c_int, [_p, _sz, _p]),
        "tt_block_attn_workspace_size": (_sz, [ctypes.POINTER(AttnDesc)]),
        "tt_block_attn": (ctypes.c_int, [ctypes.POINTER(AttnDesc), _p, _p, _p, _p, _p, _p, _p, _p,
                                         _p, _sz, _p]),
        "tt_block_attn_error": (ctypes.c_int, [_p, ctypes.POINTER(_i32), _p]),
        "tt_block_attn_ex": (ctypes.c_int, [ctypes.POINTER(AttnDesc), ctypes.POINTER(AttnOpts), _p,
                                            _p, _p, _p, _p, _p, _p, _p, _p, _sz, _p]),
        "tt_attn_lse_combine": (ctypes.c_int, [_i32, _i32, _i32, _i32, _p, _p, _p, _p, _p, _p,
                                               _p]),
        "tt_adaln_single": (ctypes.c_int, [ctypes.POINTER(AdalnDesc), _p, _p, _p, _p, _p, _p, _p,
                                           _p, _p, _p]),
        "tt_confidence_unmask_workspace_size": (_sz, [ctypes.POINTER(UnmaskDesc)]),
        "tt_confidence_unmask": (ctypes.c_int, [ctypes.POINTER(UnmaskDesc), _p, _p, _p, _p, _p, _p,
                                                _i32, _p, _sz, _p]),
        "tt_confidence_unmask_error": (ctypes.c_int, [_p, ctypes.POINTER(_i32), _p]),
        "tt_block_init": (ctypes.c_int, [ctypes.POINTER(UnmaskDesc), _p, _p, _p, _p, _p]),
        "tt_denoise_block_loop_workspace_size": (_sz, [ctypes.POINTER(UnmaskDesc)]),
        "tt_denoise_block_loop": (ctypes.c_int, [ctypes.POINTER(UnmaskDesc), _i32, _i32, _i32, _p,
                                                 _p, _p, _p, _p, _p, _p, _p, _sz, _p, _i32,
                                                 ctypes.POINTER(_i32)]),
        "tt_synth_logits": (ctypes.c_int, [ctypes.c_uint64, _i32, _i32, _i32, _i32, ctypes.c_int,
                                           ctypes.c_float, ctypes.c_uint64, _p, _p]),
        "tt_synth_logits_producer": (ctypes.c_int, [_p, _i32, _p, _p, _p, _p]),
        "tt_kv_append": (ctypes.c_int, [ctypes.POINTER(KvDesc), _p, _p, _p, _p, _p, _p, _p, _p]),
        "tt_mamba_state_seed": (ctypes.c_int, [ctypes.POINTER(StateDesc), _p, _p, _p, _p]),
        "tt_generate_blocks_workspace_size": (_sz, [ctypes.POINTER(UnmaskDesc)]),
        "tt_generate_blocks": (ctypes.c_int, [ctypes.POINTER(UnmaskDesc), ctypes.POINTER(KvDesc),
                                              ctypes.POINTER(GenerateParams), _p, _p, _p, _p,
                                              _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p, _p,
                                              _sz, _p, ctypes.POINTER(_i32)]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(s: int) -> str:
    try:
        return load().tt_status_string(int(s)).decode()
    except Exception:  # library unavailable while formatting an error
        return f"status {s}"


def last_error() -> str:
    return load().tt_last_error().decode()


def check(status: int):
    if status != TT_OK:
        raise TTError(status, last_error())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, ndim: Optional[int] = None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")


class Workspace:
    """A zeroed device workspace (uint8 tensor) sized by a *_workspace_size query."""

    def __init__(self, nbytes: int, device=None):
        if nbytes == 0:
            raise TTError(TT_ERR_INVALID_ARG, last_error() or "workspace size query failed")
        self.tensor = torch.zeros(int(nbytes) + 256, dtype=torch.uint8, device=device or "cuda")
        off = (-self.tensor.data_ptr()) % 256
        self.view = self.tensor[off:off + int(nbytes)]
        self.nbytes = int(nbytes)

    @property
    def ptr(self):
        return ctypes.c_void_p(self.view.data_ptr())


# ------------------------------------------------------------------ attention
def attn_desc(q, k_ctx, v_ctx, k_blk, v_blk, out, scale: float = 0.0) -> AttnDesc:
    B, S, Hq, d = q.shape
    Hkv, Lmax = k_ctx.shape[1], k_ctx.shape[2]
    desc = AttnDesc(B=B, S=S, Hq=Hq, Hkv=Hkv, d=d, Lmax=Lmax, scale=float(scale))
    desc.q_strides = _i64x4(*q.stride())
    desc.kctx_strides = _i64x4(*k_ctx.stride())
    desc.vctx_strides = _i64x4(*v_ctx.stride())
    desc.kblk_strides = _i64x4(*k_blk.stride())
    desc.vblk_strides = _i64x4(*v_blk.stride())
    desc.o_strides = _i64x4(*out.stride())
    return desc


def block_attn_workspace_size(desc: AttnDesc) -> int:
    return int(load().tt_block_attn_workspace_size(ctypes.byref(desc)))


def block_attn(q, k_ctx, v_ctx, ctx_lens, k_blk, v_blk, out=None, lse=None, scale: float = 0.0,
               workspace: Optional[Workspace] = None, stream=None):
    """Block-query attention (tt_block_attn).  bf16 tensors, ctx_lens int32[B].

    Returns out [B,S,Hq,d] bf16 (and writes lse [B,Hq,S] fp32 when given).
    """
    for t, n, nd in ((q, "q", 4), (k_ctx, "k_ctx", 4), (v_ctx, "v_ctx", 4), (k_blk, "k_blk", 4),
                     (v_blk, "v_blk", 4)):
        _need(t, n, torch.bfloat16, nd)
    _need(ctx_lens, "ctx_lens", torch.int32, 1)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    _need(out, "out", torch.bfloat16, 4)
    if lse is not None:
        _need(lse, "lse", torch.float32, 3)
    desc = attn_desc(q, k_ctx, v_ctx, k_blk, v_blk, out, scale)
    if workspace is None:
        workspace = Workspace(block_attn_workspace_size(desc), q.device)
    check(load().tt_block_attn(ctypes.byref(desc), _ptr(q), _ptr(k_ctx), _ptr(v_ctx),
                               _ptr(ctx_lens), _ptr(k_blk), _ptr(v_blk), _ptr(out), _ptr(lse),
                               workspace.ptr, workspace.nbytes, _stream(stream)))
    return out


def block_attn_ex(q, k_ctx, v_ctx, ctx_lens, k_blk, v_blk, keys: int = TT_KEYS_ALL,
                  block_table=None, n_pages: int = 0, q_scale=None, q_shift=None, o_gate=None,
                  out=None, lse=None, scale: float = 0.0, workspace: Optional[Workspace] = None,
                  stream=None):
    """Block-query attention with options (tt_block_attn_ex).

    keys: TT_KEYS_ALL / TT_KEYS_PREFIX / TT_KEYS_BLOCK.  block_table int32 [B, max_pages]
    selects the paged cache: k_ctx / v_ctx are then pools [n_pages, Hkv, 64, d].
    q_scale, q_shift, o_gate: fp32 [B, Hq, d] adaLN-single modulation.
    """
    for t, n, nd in ((q, "q", 4), (k_ctx, "k_ctx", 4), (v_ctx, "v_ctx", 4), (k_blk, "k_blk", 4),
                     (v_blk, "v_blk", 4)):
        _need(t, n, torch.bfloat16, nd)
    _need(ctx_lens, "ctx_lens", torch.int32, 1)
    for t, n in ((q_scale, "q_scale"), (q_shift, "q_shift"), (o_gate, "o_gate")):
        if t is not None:
            _need(t, n, torch.float32, 3)
            if not t.is_contiguous():
                raise ValueError(f"{n} must be contiguous [B, Hq, d]")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    desc = attn_desc(q, k_ctx, v_ctx, k_blk, v_blk, out, scale)
    opts = AttnOpts(keys=int(keys))
    if block_table is not None:
        _need(block_table, "block_table", torch.int32, 2)
        opts.block_table = block_table.data_ptr()
        opts.max_pages = block_table.shape[1]
        opts.n_pages = int(n_pages) if n_pages else k_ctx.shape[0]
        desc.Lmax = opts.max_pages * 64
        desc.Hkv = k_ctx.shape[1]
    for name, t in (("q_scale", q_scale), ("q_shift", q_shift), ("o_gate", o_gate)):
        if t is not None:
            setattr(opts, name, t.data_ptr())
    if workspace is None:
        workspace = Workspace(block_attn_workspace_size(desc), q.device)
    check(load().tt_block_attn_ex(ctypes.byref(desc), ctypes.byref(opts), _ptr(q), _ptr(k_ctx),
                                  _ptr(v_ctx), _ptr(ctx_lens), _ptr(k_blk), _ptr(v_blk), _ptr(out),
                                  _ptr(lse), workspace.ptr, workspace.nbytes, _stream(stream)))
    return out


def attn_lse_combine(o1, lse1, o2, lse2, out=None, lse_out=None, stream=None):
    """Joins two attention results over disjoint key sets (tt_attn_lse_combine)."""
    B, S, Hq, d = o1.shape
    for t in (o1, o2):
        _need(t, "o", torch.bfloat16, 4)
        if not t.is_contiguous():
            raise ValueError("o1 and o2 must be contiguous")
    if out is None:
        out = torch.empty_like(o1)
    check(load().tt_attn_lse_combine(B, S, Hq, d, _ptr(o1), _ptr(lse1), _ptr(o2), _ptr(lse2),
                                     _ptr(out), _ptr(lse_out), _stream(stream)))
    return out


def adaln_single(t, w1, b1, w2, b2, embed, layer: int, stream=None):
    """adaLN-single shift, scale and gate of one layer (tt_adaln_single); fp32 tensors.

    t [B]; w1 [Dh, F]; b1 [Dh]; w2 [3N, Dh]; b2 [3N]; embed [layers, 3N].
    Returns (shift, scale, gate), each [B, N].
    """
    for x, n in ((t, "t"), (w1, "w1"), (b1, "b1"), (w2, "w2"), (b2, "b2"), (embed, "embed")):
        _need(x, n, torch.float32)
        if not x.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    B, (Dh, F), N = t.shape[0], w1.shape, w2.shape[0] // 3
    outs = [torch.empty((B, N), dtype=torch.float32, device=t.device) for _ in range(3)]
    desc = AdalnDesc(B=B, F=F, Dh=Dh, N=N, layer=int(layer), n_layers=embed.shape[0])
    check(load().tt_adaln_single(ctypes.byref(desc), _ptr(t), _ptr(w1), _ptr(b1), _ptr(w2),
                                 _ptr(b2), _ptr(embed), _ptr(outs[0]), _ptr(outs[1]),
                                 _ptr(outs[2]), _stream(stream)))
    return tuple(outs)


def block_attn_noalloc(q, k_ctx, v_ctx, ctx_lens, k_blk, v_blk, out=None, lse=None,
                      scale: float = 0.0, stream=None):
    """tt_block_attn_noalloc: block attention with the library's fixed scratch.

    For callers that cannot allocate device memory: no workspace argument, and no
    allocation inside the call.  Calls must not overlap on the GPU.
    """
    lib = load()
    fn = lib.tt_block_attn_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(AttnDesc), _p, _p, _p, _p, _p, _p, _p, _p, _p]
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    desc = attn_desc(q, k_ctx, v_ctx, k_blk, v_blk, out, scale)
    check(fn(ctypes.byref(desc), _ptr(q), _ptr(k_ctx), _ptr(v_ctx), _ptr(ctx_lens), _ptr(k_blk),
             _ptr(v_blk), _ptr(out), _ptr(lse), _stream(stream)))
    return out


# ------------------------------------------------------------------ unmasking
def unmask_desc(B, S, V, dtype, temperature, threshold, mask_token_id, row_stride=0) -> UnmaskDesc:
    return UnmaskDesc(B=B, S=S, V=V, logits_dtype=dtype, logits_row_stride=row_stride,
                      temperature=float(temperature), threshold=float(threshold),
                      mask_token_id=int(mask_token_id))


def _logits_dtype(logits: torch.Tensor) -> int:
    if logits.dtype == torch.float32:
        return TT_F32
    if logits.dtype == torch.bfloat16:
        return TT_BF16
    raise TypeError("logits must be float32 or bfloat16")


def _row_stride(logits: torch.Tensor) -> int:
    B, S, V = logits.shape
    rs = logits.stride(1) if S > 1 else logits.stride(0)
    if logits.stride(2) != 1 or (B > 1 and S > 1 and logits.stride(0) != S * rs):
        raise ValueError("logits must be [B,S,V] with a uniform row stride and contiguous V")
    return rs


def confidence_unmask_workspace_size(desc: UnmaskDesc) -> int:
    return int(load().tt_confidence_unmask_workspace_size(ctypes.byref(desc)))


def confidence_unmask(logits, tokens, is_masked, temperature: float, threshold: float,
                      mask_token_id: int, force_commit_all: bool = False, conf=None,
                      committed_now=None, remaining=None, workspace: Optional[Workspace] = None,
                      stream=None) -> dict:
    """One confidence-unmasking step (tt_confidence_unmask); tokens/is_masked updated in place."""
    if logits.dim() != 3:
        raise ValueError("logits must be [B,S,V]")
    B, S, V = logits.shape
    _need(tokens, "tokens", torch.int32, 2)
    _need(is_masked, "is_masked", torch.uint8, 2)
    dev = logits.device
    conf = torch.empty((B, S), dtype=torch.float32, device=dev) if conf is None else conf
    committed_now = (torch.empty((B, S), dtype=torch.uint8, device=dev)
                     if committed_now is None else committed_now)
    remaining = torch.empty((B,), dtype=torch.int32, device=dev) if remaining is None else remaining
    desc = unmask_desc(B, S, V, _logits_dtype(logits), temperature, threshold, mask_token_id,
                       _row_stride(logits))
    if workspace is None:
        workspace = Workspace(confidence_unmask_workspace_size(desc), dev)
    check(load().tt_confidence_unmask(ctypes.byref(desc), _ptr(logits), _ptr(tokens),
                                      _ptr(is_masked), _ptr(conf), _ptr(committed_now),
                                      _ptr(remaining), int(bool(force_commit_all)), workspace.ptr,
                                      workspace.nbytes, _stream(stream)))
    return dict(tokens=tokens, is_masked=is_masked, conf=conf, committed_now=committed_now,
                remaining=remaining)


# ------------------------------------------------------------------ loop and synthetic logits
def synth_logits(seed: int, step: int, B: int, S: int, V: int, sigma: float, spike_threshold: int,
                 dtype: int = TT_BF16, out=None, stream=None):
    """Counter-based synthetic logits on the device (tt_synth_logits)."""
    if out is None:
        out = torch.empty((B, S, V), dtype=torch.bfloat16 if dtype == TT_BF16 else torch.float32,
                          device="cuda")
    check(load().tt_synth_logits(int(seed), int(step), B, S, V, int(dtype), float(sigma),
                                 int(spike_threshold), _ptr(out), _stream(stream)))
    return out


def synth_params(seed: int, B: int, S: int, V: int, dtype: int, sigma: float,
                 thresholds) -> SynthParams:
    p = SynthParams(seed=int(seed), B=B, S=S, V=V, dtype=int(dtype), sigma=float(sigma))
    thr = list(thresholds)
    for i in range(SYNTH_MAX_STEPS):
        p.spike_threshold[i] = int(thr[min(i, len(thr) - 1)]) if thr else 0
    return p


def block_init(tokens, is_masked, mask_token_id: int, steps_used=None, committed_step=None,
               stream=None):
    """Starts a block on the device (tt_block_init): all positions masked."""
    _need(tokens, "tokens", torch.int32, 2)
    _need(is_masked, "is_masked", torch.uint8, 2)
    B, S = tokens.shape
    desc = unmask_desc(B, S, 1, TT_F32, 1.0, 0.0, mask_token_id)
    check(load().tt_block_init(ctypes.byref(desc), _ptr(tokens), _ptr(is_masked), _ptr(steps_used),
                               _ptr(committed_step), _stream(stream)))


def denoise_block_loop_workspace_size(desc: UnmaskDesc) -> int:
    return int(load().tt_denoise_block_loop_workspace_size(ctypes.byref(desc)))


def denoise_block_loop(B: int, S: int, V: int, logits_dtype: int, temperature: float,
                       threshold: float, mask_token_id: int, steps_per_block: int,
                       tokens, is_masked, steps_used, committed_step=None, logits_buf=None,
                       producer: Optional[Callable] = None, synth: Optional[SynthParams] = None,
                       start_step: int = 0, stop_step: int = 0, timeout_ms: int = 60000,
                       workspace: Optional[Workspace] = None, stream=None) -> int:
    """In-block loop (tt_denoise_block_loop); returns the number of steps run.

    Exactly one of ``producer`` (a Python callable ``f(step, logits_buf)`` that
    fills the logits tensor on the current stream) or ``synth`` (parameters of
    the library's own synthetic producer) gives each step's logits.
    """
    lib = load()
    dt = torch.bfloat16 if logits_dtype == TT_BF16 else torch.float32
    if logits_buf is None:
        logits_buf = torch.empty((B, S, V), dtype=dt, device="cuda")
    desc = unmask_desc(B, S, V, logits_dtype, temperature, threshold, mask_token_id)
    if workspace is None:
        workspace = Workspace(denoise_block_loop_workspace_size(desc))
    keep = []
    if synth is not None:
        fn_ptr = ctypes.cast(lib.tt_synth_logits_producer, _p)
        user = ctypes.cast(ctypes.pointer(synth), _p)
    elif producer is not None:
        def _cb(_user, step, _tok, _msk, _out, _stream_handle):
            try:
                producer(int(step), logits_buf)
                return TT_OK
            except Exception:  # reported as TT_ERR_CALLBACK by the loop
                return TT_ERR_INTERNAL
        cb = LOGITS_FN(_cb)
        keep.append(cb)
        fn_ptr = ctypes.cast(cb, _p)
        user = None
    else:
        raise ValueError("need producer or synth")
    steps_run = _i32(0)
    status = lib.tt_denoise_block_loop(ctypes.byref(desc), steps_per_block, start_step, stop_step,
                                       fn_ptr, user, _ptr(logits_buf), _ptr(tokens),
                                       _ptr(is_masked), _ptr(steps_used), _ptr(committed_step),
                                       workspace.ptr, workspace.nbytes, _stream(stream),
                                       int(timeout_ms), ctypes.byref(steps_run))
    del keep
    check(status)
    return int(steps_run.value)


# ------------------------------------------------------------------ block append
def kv_append(k_ctx: list, v_ctx: list, ctx_lens, k_blk: list, v_blk: list, active=None,
              overflow=None, stream=None):
    """Appends the committed block's K/V of every layer to its cache (tt_kv_append).

    k_ctx/v_ctx: per layer bf16 [B,Hkv,Lmax,d]; k_blk/v_blk: per layer bf16 [B,S,Hkv,d];
    ctx_lens int32[B] is advanced in place; active uint8[B] or None; overflow int32[1]
    or None counts sequences whose block did not fit.
    """
    n = len(k_ctx)
    if not (n == len(v_ctx) == len(k_blk) == len(v_blk)) or not 1 <= n <= KV_MAX_LAYERS:
        raise ValueError(f"need 1..{KV_MAX_LAYERS} layers, the same count in each list")
    for lst, name in ((k_ctx, "k_ctx"), (v_ctx, "v_ctx"), (k_blk, "k_blk"), (v_blk, "v_blk")):
        for t in lst:
            _need(t, name, torch.bfloat16, 4)
    _need(ctx_lens, "ctx_lens", torch.int32, 1)
    if active is not None:
        _need(active, "active", torch.uint8, 1)
    if overflow is not None:
        _need(overflow, "overflow", torch.int32, 1)
    B, Hkv, Lmax, d = k_ctx[0].shape
    S = k_blk[0].shape[1]
    for lst in (k_ctx, v_ctx):
        for t in lst:
            if tuple(t.shape) != (B, Hkv, Lmax, d) or t.stride() != k_ctx[0].stride():
                raise ValueError("every cache must have the first cache's shape and strides")
    for lst in (k_blk, v_blk):
        for t in lst:
            if tuple(t.shape) != (B, S, Hkv, d) or t.stride() != k_blk[0].stride():
                raise ValueError("every block must have shape [B,S,Hkv,d] and equal strides")
    desc = KvDesc(B=B, S=S, Hkv=Hkv, d=d, Lmax=Lmax, n_layers=n)
    desc.ctx_strides = _i64x4(*k_ctx[0].stride())
    desc.blk_strides = _i64x4(*k_blk[0].stride())
    arr = ctypes.c_void_p * n
    ptrs = [arr(*[t.data_ptr() for t in lst]) for lst in (k_ctx, v_ctx, k_blk, v_blk)]
    check(load().tt_kv_append(ctypes.byref(desc), ptrs[0], ptrs[1], _ptr(ctx_lens), ptrs[2],
                              ptrs[3], _ptr(active), _ptr(overflow), _stream(stream)))


# ------------------------------------------------------------------ Mamba-2 state seeding
def mamba_state_seed(src: list, dst: list, active=None, stream=None):
    """Seeds the denoiser's Mamba-2 states from the context tower's (tt_mamba_state_seed).

    src, dst: lists over layers of lists over parts (e.g. [conv, ssm]) of device
    tensors [B, ...], each part with the same shape and strides in every layer;
    active uint8[B] or None.
    """
    n_layers, n_parts = len(src), len(src[0])
    if len(dst) != n_layers or any(len(x) != n_parts for x in src + dst):
        raise ValueError("src and dst need the same layers and parts")
    if not 1 <= n_layers <= STATE_MAX_LAYERS or not 1 <= n_parts <= STATE_MAX_PARTS:
        raise ValueError("too many layers or parts")
    B = src[0][0].shape[0]
    desc = StateDesc(B=B, n_layers=n_layers, n_parts=n_parts)
    for p in range(n_parts):
        s0, d0 = src[0][p], dst[0][p]
        for layer in range(n_layers):
            for t, ref in ((src[layer][p], s0), (dst[layer][p], d0)):
                if not t.is_cuda or t.shape != ref.shape or t.stride() != ref.stride() \
                        or t.dtype != ref.dtype or not t[0].is_contiguous():
                    raise ValueError("each part needs one shape, dtype and stride in every layer, "
                                     "with each sequence's state contiguous")
        desc.bytes[p] = s0[0].numel() * s0.element_size()
        desc.src_stride[p] = s0.stride(0) * s0.element_size()
        desc.dst_stride[p] = d0.stride(0) * d0.element_size()
    arr = ctypes.c_void_p * (n_layers * n_parts)
    sp = arr(*[src[l][p].data_ptr() for l in range(n_layers) for p in range(n_parts)])
    dp = arr(*[dst[l][p].data_ptr() for l in range(n_layers) for p in range(n_parts)])
    check(load().tt_mamba_state_seed(ctypes.byref(desc), sp, dp, _ptr(active), _stream(stream)))


# ------------------------------------------------------------------ block-by-block generation
def _kv_desc(k_ctx: list, k_blk: list) -> KvDesc:
    B, Hkv, Lmax, d = k_ctx[0].shape
    desc = KvDesc(B=B, S=k_blk[0].shape[1], Hkv=Hkv, d=d, Lmax=Lmax, n_layers=len(k_ctx))
    desc.ctx_strides = _i64x4(*k_ctx[0].stride())
    desc.blk_strides = _i64x4(*k_blk[0].stride())
    return desc


def generate_blocks(logits_fn: Callable, kv_fn: Callable, V: int, logits_dtype: int,
                    temperature: float, threshold: float, mask_token_id: int,
                    steps_per_block: int, max_new_tokens: int, eos_token_id: int,
                    k_ctx: list, v_ctx: list, ctx_lens, k_blk: list, v_blk: list,
                    out_tokens, gen_len, active, steps_total=None, overflow=None,
                    timeout_ms: int = 60000, stream=None) -> int:
    """Block-by-block generation (tt_generate_blocks); returns the number of blocks run.

    logits_fn(block, step, logits_buf) fills the [B,S,V] logits on the current
    stream; kv_fn(block, tokens, active, k_blk, v_blk) fills the per-layer block
    K/V tensors.  out_tokens int32[B,max_new], gen_len int32[B], active uint8[B]
    (in/out), steps_total int32[B] and overflow int32[1] (optional) are device
    tensors updated in place; the caches and ctx_lens as for kv_append.
    """
    lib = load()
    B, S = k_blk[0].shape[0], k_blk[0].shape[1]
    dt = torch.bfloat16 if logits_dtype == TT_BF16 else torch.float32
    logits_buf = torch.empty((B, S, V), dtype=dt, device="cuda")
    desc = unmask_desc(B, S, V, logits_dtype, temperature, threshold, mask_token_id)
    kdesc = _kv_desc(k_ctx, k_blk)
    params = GenerateParams(max_new_tokens=max_new_tokens, eos_token_id=eos_token_id,
                            steps_per_block=steps_per_block, timeout_ms=timeout_ms)
    ws = Workspace(int(lib.tt_generate_blocks_workspace_size(ctypes.byref(desc))))

    def _logits(_user, block, step, _tok, _msk, _out, _stream):
        try:
            logits_fn(int(block), int(step), logits_buf)
            return TT_OK
        except Exception:  # reported as TT_ERR_CALLBACK
            return TT_ERR_INTERNAL

    tokens_view = {}

    def _kv(_user, block, tok_ptr, act_ptr, _kb, _vb, _stream):
        try:
            if "t" not in tokens_view:
                # the library's block tokens [B, S] (device), wrapped without a copy
                tokens_view["t"] = _device_int32(tok_ptr, (B, S))
            kv_fn(int(block), tokens_view["t"], active, k_blk, v_blk)
            return TT_OK
        except Exception:
            return TT_ERR_INTERNAL

    cb_l, cb_k = BLOCK_LOGITS_FN(_logits), BLOCK_KV_FN(_kv)
    arr = ctypes.c_void_p * len(k_ctx)
    ptrs = [arr(*[t.data_ptr() for t in lst]) for lst in (k_ctx, v_ctx, k_blk, v_blk)]
    blocks = _i32(0)
    status = lib.tt_generate_blocks(ctypes.byref(desc), ctypes.byref(kdesc), ctypes.byref(params),
                                    ctypes.cast(cb_l, _p), None, ctypes.cast(cb_k, _p), None,
                                    _ptr(logits_buf), ptrs[0], ptrs[1], _ptr(ctx_lens), ptrs[2],
                                    ptrs[3], _ptr(out_tokens), _ptr(gen_len), _ptr(active),
                                    _ptr(steps_total), _ptr(overflow), ws.ptr, ws.nbytes,
                                    _stream(stream), ctypes.byref(blocks))
    check(status)
    return int(blocks.value)


def _device_int32(ptr, shape):
    """A torch int32 tensor over device memory owned by the library (no copy)."""
    n = 1
    for x in shape:
        n *= x

    class _Cuda:
        __cuda_array_interface__ = {"shape": tuple(shape), "typestr": "<i4",
                                    "data": (int(ptr), False), "version": 3, "strides": None}
    return torch.as_tensor(_Cuda(), device="cuda")


def exported_symbols() -> list:
    """Names of the entry points this binding expects libtt.so to export."""
    return ["tt_status_string", "tt_last_error", "tt_abi_version", "tt_workspace_zero",
            "tt_block_attn_workspace_size", "tt_block_attn", "tt_block_attn_error",
            "tt_block_attn_noalloc",
            "tt_confidence_unmask_workspace_size",
            "tt_confidence_unmask", "tt_confidence_unmask_error", "tt_block_init", "tt_denoise_block_loop_workspace_size",
            "tt_denoise_block_loop",
            "tt_synth_logits", "tt_synth_logits_producer", "tt_kv_append",
            "tt_mamba_state_seed", "tt_generate_blocks_workspace_size", "tt_generate_blocks",
            "tt_block_attn_ex", "tt_attn_lse_combine", "tt_adaln_single"]
