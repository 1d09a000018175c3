"""Seeded synthetic inputs for the TwoTower denoiser step (test and bench plumbing).

This module is the one piece shared by the fp64 oracle side and the CUDA side: it
only draws numbers.  It holds none of the method's arithmetic (no attention, no
softmax, no argmax, no commit rule).

Two generators:

* Static tensors (Q, K, V, context lengths): numpy PCG64 normals, rounded
  round-to-nearest-even to bf16 and kept as raw ``uint16`` bit patterns.  Each
  tensor role draws from its own stream ``SeedSequence([seed, role])``.

* Per-step vocabulary logits (the stand-in for the denoiser forward that the
  block loop calls once per step): a counter-based generator built on the
  SplitMix64 output function (Steele, Lea & Flood, "Fast splittable pseudorandom
  number generators", OOPSLA 2014; finaliser constants of Stafford's "Mix13").
  Word ``n`` of a stream with key ``k`` is ``mix64(k + (n+1)*GAMMA)``.  Each
  logit sums twelve 16-bit uniforms (three words): an Irwin-Hall(12) variate,
  which has mean 6 and variance 1, so ``z = (sum - 6*65536) * sigma / 65536`` is
  approximately N(0, sigma^2) with lighter tails, and is exact in fp32.  On a
  row chosen with probability ``p`` a spike of +8 is added at one token.  The
  CUDA library carries its own implementation of the same definition
  (``tt_synth_logits``); the two are checked bit-for-bit against each other.

Workload recipes follow the decoding configurations the TwoTower pages describe
(block_size 16, temperature 0.1, confidence threshold 0.8, mask token 3; see
"NVIDIA发布Nemotron两塔模型" (889990.xyz), the code example) with the head and
vocabulary shapes of a Nemotron-3-Nano-style backbone: Hq=32, Hkv=2, d=128,
V=131072.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_TAG_LOGITS = 0x6C6F67697473  # "logits"
_TAG_SPIKE = 0x7370696B65  # "spike"
SPIKE_MAGNITUDE = 8.0

# stream ids of the static tensors
ROLE_Q, ROLE_KCTX, ROLE_VCTX, ROLE_KBLK, ROLE_VBLK, ROLE_LENS, ROLE_LOGITS = range(7)

_U64 = np.uint64
_MASK64 = (1 << 64) - 1


# ----------------------------------------------------------------------------- bf16
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); returns uint16 bits."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact decode of bf16 bit patterns to float32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------------------- splitmix64
def mix64_int(z: int) -> int:
    """SplitMix64 output function on a Python int (mod 2^64)."""
    z &= _MASK64
    z = ((z ^ (z >> 30)) * _M1) & _MASK64
    z = ((z ^ (z >> 27)) * _M2) & _MASK64
    return z ^ (z >> 31)


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function, elementwise on uint64 arrays (wrapping arithmetic)."""
    z = z.astype(_U64, copy=True)
    z ^= z >> _U64(30)
    z *= _U64(_M1)
    z ^= z >> _U64(27)
    z *= _U64(_M2)
    z ^= z >> _U64(31)
    return z


def stream_key(seed: int, step: int) -> int:
    """Key of the logits stream for (seed, step)."""
    k0 = mix64_int((seed ^ _TAG_LOGITS) & _MASK64)
    return mix64_int(k0 + ((step + 1) * GAMMA))


def spike_threshold(p: float) -> int:
    """Integer threshold on the high 32 bits of the spike word: spike iff hi < threshold."""
    if not (0.0 <= p <= 1.0):
        raise ValueError("spike probability must lie in [0, 1]")
    return min(int(math.floor(p * 4294967296.0)), 4294967296)


def spike_draws(seed: int, step: int, n_rows: int, V: int, p: float):
    """Per-row (has_spike bool[n_rows], spike_token int64[n_rows])."""
    key = stream_key(seed, step)
    skey = mix64_int(key ^ _TAG_SPIKE)
    rows = np.arange(n_rows, dtype=_U64)
    w = mix64(_U64(skey) + (rows + _U64(1)) * _U64(GAMMA))
    hi = (w >> _U64(32)).astype(np.int64)
    lo = (w & _U64(0xFFFFFFFF)).astype(np.int64)
    return hi < spike_threshold(p), lo % V


def counter_logits_f32(seed: int, step: int, B: int, S: int, V: int, sigma: float,
                       spike_p: float = 0.0, rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Counter-generated logits as float32 [n_rows, V] (before any bf16 rounding).

    ``rows`` selects flattened row indices b*S+s (default: all B*S rows).
    """
    sig = np.float32(sigma / 65536.0)
    if float(sig) * 65536.0 != sigma:
        raise ValueError("sigma/65536 must be exact in fp32")
    key = _U64(stream_key(seed, step))
    all_rows = np.arange(B * S) if rows is None else np.asarray(rows, dtype=np.int64)
    has_spike, spike_tok = spike_draws(seed, step, B * S, V, spike_p)
    out = np.empty((len(all_rows), V), dtype=np.float32)
    v = np.arange(V, dtype=_U64)
    for i, r in enumerate(all_rows):
        acc = np.zeros(V, dtype=np.int64)
        for j in range(3):
            n = (_U64(r) * _U64(V) + v) * _U64(3) + _U64(j)
            w = mix64(key + (n + _U64(1)) * _U64(GAMMA))
            for lane in range(4):
                acc += ((w >> _U64(16 * lane)) & _U64(0xFFFF)).astype(np.int64)
        z = (acc - 6 * 65536).astype(np.float32) * sig
        if has_spike[r]:
            z[spike_tok[r]] += np.float32(SPIKE_MAGNITUDE)
        out[i] = z
    return out


def counter_logits(seed: int, step: int, B: int, S: int, V: int, sigma: float,
                   spike_p: float = 0.0, dtype: str = "bf16",
                   rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Logits [B,S,V] (or [len(rows),V]) as float32 ("f32") or bf16 bits uint16 ("bf16")."""
    z = counter_logits_f32(seed, step, B, S, V, sigma, spike_p, rows)
    if rows is None:
        z = z.reshape(B, S, V)
    if dtype == "f32":
        return z
    if dtype == "bf16":
        return bf16_bits(z)
    raise ValueError(dtype)


# ----------------------------------------------------------------------------- static tensors
def _rng(seed: int, role: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, role])))


def normal_bf16(seed: int, role: int, shape, std: float = 1.0) -> np.ndarray:
    """bf16 bits of N(0, std^2) draws (PCG64 stream (seed, role)), rounded RNE."""
    g = _rng(seed, role)
    x = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return bf16_bits(x)


@dataclass
class AttnShape:
    B: int
    S: int
    Hq: int
    Hkv: int
    d: int
    Lmax: int
    lens: Optional[list] = None  # per-sequence prefix lengths (None: uniform Lmax)
    lens_range: Optional[tuple] = None  # (lo, hi) inclusive: draw uniform integers


def ctx_lens_for(shape: AttnShape, seed: int) -> np.ndarray:
    if shape.lens is not None:
        lens = np.asarray(shape.lens, dtype=np.int32)
    elif shape.lens_range is not None:
        lo, hi = shape.lens_range
        lens = _rng(seed, ROLE_LENS).integers(lo, hi, size=shape.B, endpoint=True).astype(np.int32)
    else:
        lens = np.full(shape.B, shape.Lmax, dtype=np.int32)
    if lens.shape != (shape.B,) or lens.min(initial=0) < 0 or lens.max(initial=0) > shape.Lmax:
        raise ValueError("bad context lengths")
    return lens


def attn_inputs(shape: AttnShape, seed: int, nan_pad: bool = False) -> dict:
    """Q [B,S,Hq,d], K/V ctx [B,Hkv,Lmax,d], K/V blk [B,S,Hkv,d] as bf16 bits; lens int32[B].

    With ``nan_pad`` the context rows at or beyond each sequence's length hold NaN,
    so any read past the prefix shows up in the result.
    """
    B, S, Hq, Hkv, d, Lmax = shape.B, shape.S, shape.Hq, shape.Hkv, shape.d, shape.Lmax
    out = dict(
        q=normal_bf16(seed, ROLE_Q, (B, S, Hq, d)),
        k_ctx=normal_bf16(seed, ROLE_KCTX, (B, Hkv, Lmax, d)),
        v_ctx=normal_bf16(seed, ROLE_VCTX, (B, Hkv, Lmax, d)),
        k_blk=normal_bf16(seed, ROLE_KBLK, (B, S, Hkv, d)),
        v_blk=normal_bf16(seed, ROLE_VBLK, (B, S, Hkv, d)),
        ctx_lens=ctx_lens_for(shape, seed),
    )
    if nan_pad:
        for key in ("k_ctx", "v_ctx"):
            t = out[key]
            for b in range(B):
                t[b, :, out["ctx_lens"][b]:, :] = 0x7FC0  # bf16 quiet NaN
    return out


# ----------------------------------------------------------------------------- workloads
@dataclass
class Workload:
    """One synthetic decoding workload: attention shape plus unmask settings."""
    name: str
    attn: AttnShape
    V: int
    logits_dtype: str  # "f32" | "bf16"
    sigma: float
    spike_p: float
    temperature: float = 0.1
    threshold: float = 0.8
    mask_token_id: int = 3
    steps_per_block: int = 16
    n_layers: int = 6  # attention layers per denoiser step
    seed: int = 0
    extra: dict = field(default_factory=dict)


def workloads() -> dict:
    """The five synthetic configurations (tiny, default, ragged 16K, long, sweep), and a
    uniform 16K side point (B=8, every prefix 16384 keys)."""
    return {
        "tiny": Workload("tiny: B=1 L=64 S=16 Hq=4 Hkv=1 d=64 V=1024 f32",
                         AttnShape(1, 16, 4, 1, 64, 64), 1024, "f32", 3.0, 0.0),
        "default": Workload("default: B=8 L=4096 S=16 Hq=32 Hkv=2 d=128 V=131072",
                            AttnShape(8, 16, 32, 2, 128, 4096), 131072, "bf16", 2.0, 0.6),
        "ragged16k": Workload("ragged16k: B=32 L~U[1024,16384] S=16 Hq=32 Hkv=2 d=128 V=131072",
                              AttnShape(32, 16, 32, 2, 128, 16384, lens_range=(1024, 16384)),
                              131072, "bf16", 2.0, 0.6),
        "uniform16k": Workload("uniform16k: B=8 L=16384 S=16 Hq=32 Hkv=2 d=128 V=131072",
                               AttnShape(8, 16, 32, 2, 128, 16384), 131072, "bf16", 2.0, 0.6),
        "long": Workload("long: B=4 L=131072 S=16 Hq=32 Hkv=2 d=128 V=131072",
                         AttnShape(4, 16, 32, 2, 128, 131072), 131072, "bf16", 2.0, 0.6),
        "sweep": Workload("sweep: B=16 L=8192 S in {4..64} Hq=32 Hkv=2 d=128 V=131072",
                          AttnShape(16, 16, 32, 2, 128, 8192), 131072, "bf16", 2.0, 0.2,
                          extra=dict(S_values=(4, 8, 16, 32, 64), gammas=(0.5, 0.8, 0.95),
                                     spike_p_first=0.2, spike_p_last=0.9)),
    }


def sweep_spike_p(step: int, steps: int, p_first: float = 0.2, p_last: float = 0.9) -> float:
    """Spike probability growing linearly across the steps of a block."""
    if steps <= 1:
        return p_last
    return p_first + (p_last - p_first) * step / (steps - 1)
