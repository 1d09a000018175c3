"""fp64 CPU oracle for the TwoTower denoiser step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this module.  It wraps ``oracle.c`` (plain C, fp64,
compiled with gcc) through ctypes and adds the block loop, which is plain
Python around the per-step unmask.  It shares nothing with the CUDA library.

Parity status of every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants, library special cases, brute force, planted mistakes).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Callable, Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

_p = ctypes.c_void_p
_i = ctypes.c_int


def build(out_path: str = _LIB_PATH, defines: tuple = ()) -> str:
    """Compile oracle.c with gcc into a shared library; returns its path."""
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", "-Wall", "-Werror"]
    cmd += [f"-D{d}" for d in defines]
    cmd += [_SRC, "-o", out_path, "-lm"]
    subprocess.run(cmd, check=True)
    return out_path


def _needs_build(path: str) -> bool:
    return not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC)


def load(path: Optional[str] = None):
    """Load (building when stale) the oracle library; returns the ctypes handle."""
    global _lib
    if path is None:
        if _lib is not None:
            return _lib
        if _needs_build(_LIB_PATH):
            build()
        path = _LIB_PATH
    lib = ctypes.CDLL(path)
    lib.oracle_hw_threads.restype = _i
    lib.oracle_block_attn.restype = _i
    lib.oracle_block_attn.argtypes = [_i, _i, _i, _i, _i, _i, ctypes.c_double,
                                      _p, _p, _p, _p, _p, _p, _p, _p, _i]
    lib.oracle_block_attn2.restype = _i
    lib.oracle_block_attn2.argtypes = [_i, _i, _i, _i, _i, _i, ctypes.c_double, _p, _p, _p, _p,
                                       _p, _p, _p, _i, _p, _p, _p, _i]
    lib.oracle_confidence_unmask.restype = _i
    lib.oracle_confidence_unmask.argtypes = [_i, _i, _i, _i, _p, ctypes.c_double, ctypes.c_float,
                                             ctypes.c_int32, _i, _p, _p, _p, _p, _p, _p, _i]
    if path == _LIB_PATH:
        _lib = lib
    return lib


def hw_threads() -> int:
    return load().oracle_hw_threads()


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


KEYS = {"all": 0, "prefix": 1, "block": 2}


def bf16_decode(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def block_attn(q, k_ctx, v_ctx, ctx_lens, k_blk, v_blk, scale: float = 0.0,
               nthreads: int = 0, lib=None, return_threads: bool = False, keys: str = "all",
               q_scale=None, q_shift=None, o_gate=None):
    """Exact block-query attention in fp64.

    q [B,S,Hq,d], k_ctx/v_ctx [B,Hkv,Lmax,d], k_blk/v_blk [B,S,Hkv,d]: bf16 bit
    patterns (uint16).  ctx_lens int32[B].  scale <= 0 means 1/sqrt(d).
    keys: "all" (the prefix then the block, one softmax), "prefix" or "block" (one of
    the two key sets alone; a row that sees no key gets out 0 and lse -inf).
    q_scale, q_shift, o_gate ([B,Hq,d], optional): adaLN-single modulation, in fp64:
    queries q * (1 + q_scale) + q_shift, output multiplied by o_gate (the aitrends.kr
    page, technical features: scale, shift and gate per timestep in each denoiser
    layer).  Returns (out float64 [B,S,Hq,d], lse float64 [B,Hq,S]).
    """
    lib = lib or load()
    q, k_blk, v_blk = _c(q, np.uint16), _c(k_blk, np.uint16), _c(v_blk, np.uint16)
    k_ctx, v_ctx = _c(k_ctx, np.uint16), _c(v_ctx, np.uint16)
    lens = _c(ctx_lens, np.int32)
    B, S, Hq, d = q.shape
    Hkv, Lmax = k_ctx.shape[1], k_ctx.shape[2]
    out = np.empty((B, S, Hq, d), dtype=np.float64)
    lse = np.empty((B, Hq, S), dtype=np.float64)
    q64 = None
    if q_scale is not None or q_shift is not None:
        sc = np.zeros((B, Hq, d)) if q_scale is None else np.asarray(q_scale, np.float64)
        sh = np.zeros((B, Hq, d)) if q_shift is None else np.asarray(q_shift, np.float64)
        q64 = _c(bf16_decode(q) * (1.0 + sc[:, None]) + sh[:, None], np.float64)
    gate = None if o_gate is None else _c(o_gate, np.float64)
    used = lib.oracle_block_attn2(B, S, Hq, Hkv, d, Lmax, float(scale), _ptr(q), _ptr(q64),
                                  _ptr(k_ctx), _ptr(v_ctx), _ptr(lens), _ptr(k_blk), _ptr(v_blk),
                                  KEYS[keys], _ptr(gate), _ptr(out), _ptr(lse), int(nthreads))
    if used < 0:
        raise ValueError("oracle_block_attn2: invalid arguments")
    return (out, lse, used) if return_threads else (out, lse)


def lse_combine(o1, lse1, o2, lse2):
    """The softmax over the union of two disjoint key sets from the results over each
    (o [B,S,Hq,d], natural-log lse [B,Hq,S], float64): with M = max(lse1, lse2) and
    w_i = exp(lse_i - M), o = (w1 o1 + w2 o2) / (w1 + w2), lse = M + log(w1 + w2); a
    side with lse = -inf (no key) weighs nothing, and both gives o = 0, lse = -inf."""
    l1 = np.asarray(lse1, np.float64)
    l2 = np.asarray(lse2, np.float64)
    M = np.maximum(l1, l2)
    finite = np.isfinite(M)
    Ms = np.where(finite, M, 0.0)
    w1 = np.where(np.isfinite(l1), np.exp(np.where(np.isfinite(l1), l1, 0.0) - Ms), 0.0)
    w2 = np.where(np.isfinite(l2), np.exp(np.where(np.isfinite(l2), l2, 0.0) - Ms), 0.0)
    den = w1 + w2
    # [B,Hq,S] weights onto [B,S,Hq,1]
    t = lambda x: np.transpose(x, (0, 2, 1))[..., None]  # noqa: E731
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(t(den) > 0, (t(w1) * o1 + t(w2) * o2) / np.where(t(den) > 0, t(den), 1.0), 0.0)
        lse = np.where(den > 0, Ms + np.log(np.where(den > 0, den, 1.0)), -np.inf)
    return o, lse


def adaln_single(t, w1, b1, w2, b2, embed, layer: int):
    """adaLN-single modulation of one denoiser layer from the diffusion timestep.

    The pages say each denoiser layer is modulated by the diffusion timestep through
    adaLN-single, which injects a scale, shift and gate per timestep with about 1.5 M
    added parameters (aitrends.kr, "Nemotron-Labs-TwoTower-30B-A3B-Base-BF16", section
    기술적 특징; dothoosh.com, architecture bullets).  adaLN-single computes the
    modulation once from the timestep with a small network shared by all layers and
    adds a per-layer learned offset.  Reading (the pages give no further detail):
      e(t)  = [cos(t w_0), .., cos(t w_{F/2-1}), sin(t w_0), .., sin(t w_{F/2-1})],
              w_i = 10000^(-i / (F/2))   (a sinusoidal timestep embedding of size F);
      h     = SiLU(W1 e(t) + b1),  SiLU(x) = x / (1 + exp(-x))   (W1 [Dh, F]);
      m     = W2 h + b2 + embed[layer]   (W2 [3 N, Dh], embed [layers, 3 N]);
      shift, scale, gate = m[0:N], m[N:2N], m[2N:3N].
    t: [B] float timesteps.  Returns (shift, scale, gate), each float64 [B, N].
    """
    t = np.asarray(t, np.float64)
    w1 = np.asarray(w1, np.float64)
    F = w1.shape[1]
    half = F // 2
    freqs = 10000.0 ** (-np.arange(half, dtype=np.float64) / half)
    arg = t[:, None] * freqs[None, :]
    e = np.concatenate([np.cos(arg), np.sin(arg)], axis=1)
    pre = e @ w1.T + np.asarray(b1, np.float64)[None, :]
    h = pre / (1.0 + np.exp(-pre))
    m = h @ np.asarray(w2, np.float64).T + np.asarray(b2, np.float64)[None, :] + \
        np.asarray(embed, np.float64)[layer][None, :]
    N = m.shape[1] // 3
    return m[:, :N], m[:, N:2 * N], m[:, 2 * N:]


def confidence_unmask(logits, dtype: str, temperature: float, threshold: float,
                      mask_token_id: int, tokens, is_masked, force_commit_all: bool = False,
                      nthreads: int = 0, lib=None) -> dict:
    """One confidence-unmasking step (see oracle.c).  tokens/is_masked are copied.

    Returns dict(tokens, is_masked, conf, committed_now, remaining, ambiguous, threads).
    """
    lib = lib or load()
    if dtype not in ("f32", "bf16"):
        raise ValueError(dtype)
    lg = _c(logits, np.float32 if dtype == "f32" else np.uint16)
    B, S, V = lg.shape
    tok = np.array(tokens, dtype=np.int32, copy=True).reshape(B, S)
    msk = np.array(is_masked, dtype=np.uint8, copy=True).reshape(B, S)
    conf = np.empty((B, S), dtype=np.float64)
    now = np.empty((B, S), dtype=np.uint8)
    rem = np.empty((B,), dtype=np.int32)
    amb = np.empty((B, S), dtype=np.uint8)
    used = lib.oracle_confidence_unmask(B, S, V, 0 if dtype == "f32" else 1, _ptr(lg),
                                        float(temperature), float(threshold), int(mask_token_id),
                                        int(bool(force_commit_all)), _ptr(tok), _ptr(msk),
                                        _ptr(conf), _ptr(now), _ptr(rem), _ptr(amb), int(nthreads))
    if used < 0:
        raise ValueError("oracle_confidence_unmask: invalid arguments")
    return dict(tokens=tok, is_masked=msk, conf=conf, committed_now=now, remaining=rem,
                ambiguous=amb, threads=used)


def block_loop(B: int, S: int, logits_fn: Callable[[int], np.ndarray], dtype: str,
               temperature: float, threshold: float, mask_token_id: int, steps_per_block: int,
               start_step: int = 0, state: Optional[dict] = None,
               stop_step: Optional[int] = None, nthreads: int = 0, lib=None,
               active: Optional[np.ndarray] = None) -> dict:
    """In-block iteration of the denoiser step.

    A block starts as S copies of mask_token_id, all masked.  For step k in
    [start_step, stop_step) (stop_step defaults to steps_per_block): stop early
    once nothing is masked; otherwise
    take the step's logits from logits_fn(k) (the stand-in for the denoiser
    forward), run one unmask step -- forcing every remaining position to commit
    at the last step -- and count the step for each sequence that still had a
    masked position.  ``state`` (tokens, is_masked, steps_used, committed_step)
    resumes an interrupted loop.  ``active`` (bool/uint8 [B]) restricts a fresh
    block to the sequences that take part: the others start with nothing masked.
    Follows the block-by-block mechanism of the dothoosh.com article (section
    "two-tower mechanism") and the generate arguments of the 889990.xyz code
    example.
    """
    if state is None or start_step == 0:
        tokens = np.full((B, S), mask_token_id, dtype=np.int32)
        masked = np.ones((B, S), dtype=np.uint8)
        if active is not None:
            masked[np.asarray(active).reshape(B) == 0] = 0
        steps_used = np.zeros((B,), dtype=np.int32)
        committed_step = np.full((B, S), -1, dtype=np.int32)
    else:
        tokens = np.array(state["tokens"], dtype=np.int32, copy=True)
        masked = np.array(state["is_masked"], dtype=np.uint8, copy=True)
        steps_used = np.array(state["steps_used"], dtype=np.int32, copy=True)
        committed_step = np.array(state["committed_step"], dtype=np.int32, copy=True)
    ambiguous = 0
    stop = steps_per_block if stop_step is None else min(stop_step, steps_per_block)
    for k in range(start_step, stop):
        active = masked.reshape(B, S).any(axis=1)
        if not active.any():
            break
        r = confidence_unmask(logits_fn(k), dtype, temperature, threshold, mask_token_id,
                              tokens, masked, force_commit_all=(k == steps_per_block - 1),
                              nthreads=nthreads, lib=lib)
        steps_used += active.astype(np.int32)
        committed_step[r["committed_now"] == 1] = k
        tokens, masked = r["tokens"], r["is_masked"]
        ambiguous += int(r["ambiguous"].sum())
    return dict(tokens=tokens, is_masked=masked, steps_used=steps_used,
                committed_step=committed_step, ambiguous=ambiguous)


def kv_append(k_ctx: list, v_ctx: list, ctx_lens, k_blk: list, v_blk: list,
              active=None) -> dict:
    """Makes a committed block part of the context of every layer.

    For sequence b taking part (``active`` is None or active[b] != 0) with prefix
    length L_b = ctx_lens[b] and L_b + S <= Lmax: the S block rows of layer l, KV
    head g, are written after the prefix, cache row L_b + s <- block row s, and the
    prefix length becomes L_b + S.  Any other sequence keeps its cache and length;
    one taking part that does not fit is counted in ``overflow``.  Follows the
    block-by-block mechanism of the dothoosh.com article (section "two-tower
    mechanism"): each clean block becomes context for the next one.

    Caches are [B, Hkv, Lmax, d] and blocks [B, S, Hkv, d] per layer, copied as
    they are (any dtype).  Returns new caches, lengths and the overflow count.
    """
    lens = np.asarray(ctx_lens).astype(np.int64)
    B = lens.shape[0]
    S = k_blk[0].shape[1]
    Lmax = k_ctx[0].shape[2]
    out_k = [np.array(k, copy=True) for k in k_ctx]
    out_v = [np.array(v, copy=True) for v in v_ctx]
    new_lens = np.array(ctx_lens, dtype=np.int32, copy=True)
    overflow = 0
    for b in range(B):
        if active is not None and not active[b]:
            continue
        L = int(lens[b])
        if L < 0 or L + S > Lmax:
            overflow += 1
            continue
        for layer in range(len(k_ctx)):
            for s in range(S):
                for g in range(k_blk[layer].shape[2]):
                    out_k[layer][b, g, L + s, :] = k_blk[layer][b, s, g, :]
                    out_v[layer][b, g, L + s, :] = v_blk[layer][b, s, g, :]
        new_lens[b] = L + S
    return dict(k_ctx=out_k, v_ctx=out_v, ctx_lens=new_lens, overflow=overflow)


def generate_blocks(B: int, S: int, logits_fn: Callable[[int, int], np.ndarray],
                    kv_fn: Callable[[int, np.ndarray], tuple], k_ctx: list, v_ctx: list,
                    ctx_lens, dtype: str, temperature: float, threshold: float,
                    mask_token_id: int, steps_per_block: int, max_new_tokens: int,
                    eos_token_id: int = -1, active=None, out_fill: int = -1) -> dict:
    """Block-by-block generation: blocks of S positions are denoised one after another,
    and each finished block becomes context for the next.

    The pages describe this outer loop: the denoiser fills a block of masked
    positions step by step, the clean block is handed to the context tower, and the
    next block attends to the longer prefix (dothoosh.com, "فرآیند انتشار در برابر
    رمزگشایی متوالی در مدل جدید انویدیا", section on the two-tower mechanism); the
    generate call takes max_new_tokens, block_size, steps_per_block and
    eos_token_id (889990.xyz, "NVIDIA发布Nemotron两塔模型", section 训练与推理, code
    example).  Readings, where the pages are silent:

    * the number of blocks is ceil(max_new_tokens / S); positions of the last block
      past max_new_tokens are generated but not kept;
    * a sequence stops after the block in which it commits eos_token_id; its
      generated length counts the tokens up to and including the first EOS of the
      kept positions; a sequence also stops at max_new_tokens, and when its context
      cache cannot take another block (counted in ``overflow``);
    * a stopped sequence takes no part in later blocks (nothing masked, nothing
      appended); only sequences that continue get the block's K/V appended, and
      after the last block nothing is appended.

    logits_fn(block, step) gives [B,S,V] logits (the denoiser forward's stand-in);
    kv_fn(block, tokens [B,S]) gives (k list, v list) per layer [B,S,Hkv,d] for the
    committed block (the context tower's stand-in).  Returns out_tokens [B,
    max_new_tokens] (``out_fill`` where nothing was generated), gen_len [B], the
    final active flags, context lengths and caches, steps_total [B], blocks_run and
    overflow.
    """
    n_blocks = -(-max_new_tokens // S)
    act = np.ones(B, dtype=np.uint8) if active is None else np.array(active, np.uint8, copy=True)
    out = np.full((B, max_new_tokens), out_fill, dtype=np.int32)
    gen_len = np.zeros(B, dtype=np.int32)
    steps_total = np.zeros(B, dtype=np.int32)
    lens = np.array(ctx_lens, dtype=np.int32, copy=True)
    kc = [np.array(k, copy=True) for k in k_ctx]
    vc = [np.array(v, copy=True) for v in v_ctx]
    Lmax = kc[0].shape[2]
    overflow = 0
    blocks_run = 0
    ambiguous = 0
    for blk in range(n_blocks):
        if not act.any():
            break
        r = block_loop(B, S, lambda k: logits_fn(blk, k), dtype, temperature, threshold,
                       mask_token_id, steps_per_block, active=act)
        ambiguous += r["ambiguous"]
        blocks_run += 1
        keep = min(S, max_new_tokens - blk * S)
        for b in range(B):
            if not act[b]:
                continue
            toks = r["tokens"][b, :keep]
            out[b, blk * S: blk * S + keep] = toks
            steps_total[b] += r["steps_used"][b]
            hits = np.nonzero(toks == eos_token_id)[0] if eos_token_id >= 0 else []
            if len(hits):
                gen_len[b] = blk * S + int(hits[0]) + 1
                act[b] = 0
                continue
            gen_len[b] = blk * S + keep
            if gen_len[b] == max_new_tokens:
                act[b] = 0
            elif lens[b] + S > Lmax:  # the cache cannot take this block
                act[b] = 0
                overflow += 1
        if blk + 1 < n_blocks and act.any():
            kb, vb = kv_fn(blk, r["tokens"])
            a = kv_append(kc, vc, lens, kb, vb, active=act)
            kc, vc, lens = a["k_ctx"], a["v_ctx"], a["ctx_lens"]
    return dict(out_tokens=out, gen_len=gen_len, active=act, ctx_lens=lens, k_ctx=kc, v_ctx=vc,
                steps_total=steps_total, blocks_run=blocks_run, overflow=overflow,
                ambiguous=ambiguous)


def mamba_state_seed(src: list, dst: list, active=None) -> list:
    """Seeds the denoiser's Mamba-2 layers with the context tower's states.

    The pages describe the coupling: the denoiser's Mamba-2 layers take their initial
    state directly from the corresponding Mamba layer of the context tower
    (dothoosh.com, "فرآیند انتشار در برابر رمزگشایی متوالی در مدل جدید انویدیا",
    architecture bullets), that is, the context tower's conv/SSM boundary states are
    injected as the initial states of the denoiser's Mamba layers (aitrends.kr,
    "Nemotron-Labs-TwoTower-30B-A3B-Base-BF16", section 기술적 특징).  No recurrence
    is given, so this is the seeding itself: for every layer l, state part p (conv,
    SSM, ...) and sequence b taking part (``active`` None or active[b] != 0),
    dst[l][p][b] = src[l][p][b], bytes unchanged; other sequences keep their state.

    src, dst: lists over layers of lists over parts of arrays [B, ...] (any dtype).
    Returns the new destination arrays.
    """
    out = [[np.array(x, copy=True) for x in layer] for layer in dst]
    for layer in range(len(src)):
        for part in range(len(src[layer])):
            B = src[layer][part].shape[0]
            for b in range(B):
                if active is not None and not active[b]:
                    continue
                out[layer][part][b] = src[layer][part][b]
    return out
