#!/usr/bin/env python3
"""Bench of the TwoTower denoiser-step hot path on B300.

One step = one denoiser step of a block: tt_block_init (block of mask tokens),
then block-query attention for each of the denoiser's 6 attention layers (layer
i reads its own context-tower K/V cache), then one confidence-unmasking step
over the block's logits.  Inputs are synthetic, seeded and resident in HBM.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

Prints one JSON line (rank 0).  value = block-attention query tokens per second
summed over the attention layers (B*S*layers per step / step time) over all
ranks; the JSON also carries attention HBM GB/s against the measured roofline,
unmask positions/s, an end-to-end figure through the C ABI with host buffers,
and the fp64 oracle timed on the host cores on a bounded sample.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import sys
import time
from typing import Optional

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from block_mask_diffusion_tt_b300 import synth, tt  # noqa: E402

METRIC = "block-attn query-tokens/s + HBM GB/s (% roofline); unmask positions/s"
UNIT = "query-tokens/s"
NORTH_STAR_HBM_GBS = 8000.0


def measured_peaks() -> dict:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p["bf16_tflops_sustained"]), source="measured")
    except Exception:
        return dict(hbm_gbs=6400.0, bf16_tflops=1800.0, bf16_tflops_sustained=1400.0,
                    source="fallback")


def code_hash(path: str) -> str:
    """sha256 of a C/CUDA source with comments and whitespace removed, so that a
    record taken on one version of a kernel stays valid across comment edits only."""
    import hashlib
    import re
    src = open(path).read()
    src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
    src = re.sub(r"//[^\n]*", " ", src)
    return hashlib.sha256("".join(src.split()).encode()).hexdigest()


def recorded_traffic(workload: str):
    """DRAM bytes per attention call from the committed ncu capture summary
    (profiles/traffic.json), used only while the attention source is the code that
    capture measured (code_hash of attn.cu); otherwise None."""
    try:
        src = os.path.join(ROOT, "block_mask_diffusion_tt_b300", "csrc", "attn.cu")
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            rec = json.load(f)
        e = rec.get(workload)
        if e and e.get("attn_cu_code_sha256") == code_hash(src):
            return e["dram_bytes_per_call"]
    except Exception:
        pass
    return None


# ------------------------------------------------------------------ distributed plumbing
def rank_seed(w: synth.Workload, rank: int) -> int:
    """Seed of rank `rank`'s batch: every rank draws its own independent batch of the
    workload (weak scaling, no data exchanged between ranks)."""
    return w.seed + rank

class Dist:
    def __init__(self, want: int, init: bool = True):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1 and init:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend)
            self.pg = dist
        if want != self.world and self.world > 1 and self.rank == 0:
            print(f"warning: --gpus {want} but WORLD_SIZE {self.world}", file=sys.stderr)

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# ------------------------------------------------------------------ clocks
class _CtypesNvml:
    """The few read-only NVML queries the clock sampler uses, called through ctypes on
    the driver's libnvidia-ml (for hosts without the nvidia-ml-py module)."""
    NVML_CLOCK_SM = 1

    def __init__(self):
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")

    def _ok(self, r, what):
        if r != 0:
            raise RuntimeError(f"{what} returned {r}")

    def nvmlInit(self):
        self._ok(self.lib.nvmlInit_v2(), "nvmlInit_v2")

    def nvmlShutdown(self):
        self.lib.nvmlShutdown()

    def nvmlDeviceGetHandleByUUID(self, uuid: bytes):
        h = ctypes.c_void_p()
        self._ok(self.lib.nvmlDeviceGetHandleByUUID(ctypes.c_char_p(uuid), ctypes.byref(h)),
                 "nvmlDeviceGetHandleByUUID")
        return h

    def nvmlDeviceGetHandleByIndex(self, i: int):
        h = ctypes.c_void_p()
        self._ok(self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(i), ctypes.byref(h)),
                 "nvmlDeviceGetHandleByIndex_v2")
        return h

    def nvmlDeviceGetClockInfo(self, h, clock: int) -> int:
        v = ctypes.c_uint()
        self._ok(self.lib.nvmlDeviceGetClockInfo(h, ctypes.c_int(clock), ctypes.byref(v)),
                 "nvmlDeviceGetClockInfo")
        return v.value

    def nvmlDeviceGetMaxClockInfo(self, h, clock: int) -> int:
        v = ctypes.c_uint()
        self._ok(self.lib.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(clock), ctypes.byref(v)),
                 "nvmlDeviceGetMaxClockInfo")
        return v.value

    def nvmlDeviceGetPowerUsage(self, h) -> int:
        v = ctypes.c_uint()
        self._ok(self.lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(v)), "nvmlDeviceGetPowerUsage")
        return v.value

    def nvmlDeviceGetCurrentClocksThrottleReasons(self, h) -> int:
        v = ctypes.c_ulonglong()
        self._ok(self.lib.nvmlDeviceGetCurrentClocksThrottleReasons(h, ctypes.byref(v)),
                 "nvmlDeviceGetCurrentClocksThrottleReasons")
        return v.value


class ClockSampler:
    """Samples the GPU's SM clock, power and clock-event reasons during the timed region.

    Read-only NVML queries (nvidia-ml-py) from a background thread, about one per
    millisecond, so a timed region of a few milliseconds still gets samples; if NVML
    cannot be used the record says why.  `mark_start()` and `mark_end()` bracket the
    timed region; only samples taken between them count."""
    REASONS = (("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40),
               ("sw_thermal_slowdown", 0x20), ("sw_power_cap", 0x4))

    def __init__(self, device_index: int):
        import threading
        self.samples = []  # (t, sm_mhz, power_w, reasons bitmask)
        self.t0 = self.t1 = None
        self.err = None
        self.stop_ev = threading.Event()
        self.ready = threading.Event()
        self.max_mhz = None
        try:
            try:
                import pynvml
            except ImportError:  # the driver's libnvidia-ml through ctypes
                pynvml = _CtypesNvml()
            pynvml.nvmlInit()
            self.nvml = pynvml
            self.handle = self._handle(device_index)
            self.max_mhz = float(pynvml.nvmlDeviceGetMaxClockInfo(self.handle,
                                                                  pynvml.NVML_CLOCK_SM))
        except Exception as e:  # no NVML: nothing to sample
            self.nvml, self.err = None, f"nvml unavailable: {e}"
            self.ready.set()
            return
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()
        self.ready.wait(5.0)

    def _handle(self, device_index: int):
        nv = self.nvml
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            return nv.nvmlDeviceGetHandleByUUID(("GPU-" + uuid).encode())
        except Exception:
            vis = [v.strip() for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")
                   if v.strip()]
            idx = int(vis[device_index]) if device_index < len(vis) and vis[device_index].isdigit() \
                else device_index
            return nv.nvmlDeviceGetHandleByIndex(idx)

    def _run(self):
        nv, h = self.nvml, self.handle
        get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop_ev.is_set():
            try:
                t = time.perf_counter()
                sm = float(nv.nvmlDeviceGetClockInfo(h, nv.NVML_CLOCK_SM))
                pw = nv.nvmlDeviceGetPowerUsage(h) / 1000.0
                rs = int(get_reasons(h))
                self.samples.append((t, sm, pw, rs))
            except Exception as e:
                self.err = str(e)
                self.ready.set()
                return
            self.ready.set()
            time.sleep(0.001)

    def mark_start(self):
        self.t0 = time.perf_counter()

    def mark_end(self):
        self.t1 = time.perf_counter()

    def stop(self) -> dict:
        if self.nvml is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [self.err or "no nvml"]}
        self.stop_ev.set()
        self.thread.join(2.0)
        t0 = self.t0 if self.t0 is not None else -math.inf
        t1 = self.t1 if self.t1 is not None else math.inf
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        # a region shorter than the sampling period: take the samples nearest to it
        if not inside and self.samples:
            mid = 0.5 * (t0 + t1) if math.isfinite(t0) and math.isfinite(t1) else self.samples[-1][0]
            inside = sorted(self.samples, key=lambda x: abs(x[0] - mid))[:3]
        try:
            self.nvml.nvmlShutdown()
        except Exception:
            pass
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz,
                    "reasons": [self.err or "no samples"]}
        reasons = sorted({n for _, _, _, rs in inside for n, bit in self.REASONS if rs & bit})
        return {"sm_mhz": float(np.median([x[1] for x in inside])), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(inside),
                "power_w_max": float(max(x[2] for x in inside)), "source": "nvml, 1 ms"}


# ------------------------------------------------------------------ workload on the device
class DeviceWorkload:
    def __init__(self, w: synth.Workload, seed: int, device: str):
        a = w.attn
        self.w, self.a, self.dev = w, a, device
        g = torch.Generator(device=device)
        g.manual_seed(1000 + seed)

        def randn(shape):
            return torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(
                torch.bfloat16)

        self.lens_np = synth.ctx_lens_for(a, seed)
        self.lens = torch.from_numpy(self.lens_np).to(device)
        L = w.n_layers
        self.layers = []
        for _ in range(L):
            self.layers.append(dict(
                q=randn((a.B, a.S, a.Hq, a.d)), k_ctx=randn((a.B, a.Hkv, a.Lmax, a.d)),
                v_ctx=randn((a.B, a.Hkv, a.Lmax, a.d)), k_blk=randn((a.B, a.S, a.Hkv, a.d)),
                v_blk=randn((a.B, a.S, a.Hkv, a.d)),
                out=torch.empty((a.B, a.S, a.Hq, a.d), dtype=torch.bfloat16, device=device)))
        self.logits = tt.synth_logits(seed, 0, a.B, a.S, w.V, w.sigma,
                                      synth.spike_threshold(w.spike_p), tt.TT_BF16)
        self.tokens = torch.empty((a.B, a.S), dtype=torch.int32, device=device)
        self.masked = torch.empty((a.B, a.S), dtype=torch.uint8, device=device)
        self.conf = torch.empty((a.B, a.S), dtype=torch.float32, device=device)
        self.now = torch.empty((a.B, a.S), dtype=torch.uint8, device=device)
        self.remaining = torch.empty((a.B,), dtype=torch.int32, device=device)
        l0 = self.layers[0]
        self.attn_desc = tt.attn_desc(l0["q"], l0["k_ctx"], l0["v_ctx"], l0["k_blk"], l0["v_blk"],
                                      l0["out"])
        self.attn_ws = tt.Workspace(tt.block_attn_workspace_size(self.attn_desc), device)
        self.unmask_desc = tt.unmask_desc(a.B, a.S, w.V, tt.TT_BF16, w.temperature, w.threshold,
                                          w.mask_token_id)
        self.unmask_ws = tt.Workspace(tt.confidence_unmask_workspace_size(self.unmask_desc),
                                      device)
        torch.cuda.synchronize()
        self.lib = tt.load()
        # block_init, per layer the attention kernel and its split-K merge, and the
        # unmask's streaming and commit kernels
        self.launches_per_step = 1 + 2 * L + 2

    # algorithmic bytes of one attention launch: visible K/V, block K/V, Q, O
    def attn_bytes(self) -> int:
        a = self.a
        kv = int(self.lens_np.sum()) * a.Hkv * a.d * 2 * 2
        blk = a.B * a.S * a.Hkv * a.d * 2 * 2
        qo = a.B * a.S * a.Hq * a.d * 2 * 2
        return kv + blk + qo

    def attn_flops(self) -> int:
        a = self.a
        return int(4 * a.S * a.Hq * a.d * (self.lens_np.astype(np.int64) + a.S).sum())

    def unmask_bytes(self) -> int:  # every position masked at a block's first step
        a = self.a
        return a.B * a.S * self.w.V * 2 + a.B * a.S * (4 + 1 + 4 + 1 + 4) + a.B * 4

    def step(self, stream, ev_attn=None, ev_unmask=None):
        """Enqueues one denoiser step; optional event pairs bracket the attention calls
        (one pair around the layers' back-to-back calls) and the unmask call."""
        sp = ctypes.c_void_p(stream.cuda_stream)
        lib = self.lib
        tt.check(lib.tt_block_init(ctypes.byref(self.unmask_desc), tt._ptr(self.tokens),
                                   tt._ptr(self.masked), None, None, sp))
        for i, ly in enumerate(self.layers):
            if ev_attn is not None and i == 0:
                ev_attn[0].record(stream)
            tt.check(lib.tt_block_attn(ctypes.byref(self.attn_desc), tt._ptr(ly["q"]),
                                       tt._ptr(ly["k_ctx"]), tt._ptr(ly["v_ctx"]),
                                       tt._ptr(self.lens), tt._ptr(ly["k_blk"]),
                                       tt._ptr(ly["v_blk"]), tt._ptr(ly["out"]), None,
                                       self.attn_ws.ptr, self.attn_ws.nbytes, sp))
            if ev_attn is not None and i == len(self.layers) - 1:
                ev_attn[1].record(stream)
        if ev_unmask is not None:
            ev_unmask[0].record(stream)
        tt.check(lib.tt_confidence_unmask(ctypes.byref(self.unmask_desc), tt._ptr(self.logits),
                                          tt._ptr(self.tokens), tt._ptr(self.masked),
                                          tt._ptr(self.conf), tt._ptr(self.now),
                                          tt._ptr(self.remaining), 0, self.unmask_ws.ptr,
                                          self.unmask_ws.nbytes, sp))
        if ev_unmask is not None:
            ev_unmask[1].record(stream)


def run_ours(args, dist: Dist) -> dict:
    w = synth.workloads()[args.workload]
    dev = f"cuda:{dist.local}"
    torch.cuda.set_device(dist.local)
    stream = torch.cuda.Stream()
    wl = DeviceWorkload(w, seed=rank_seed(w, dist.rank), device=dev)
    a = wl.a
    clocks = ClockSampler(dist.local)
    # With graphs (the default) the step is captured once per M steps (M the largest
    # divisor of K up to 10), with event pairs inside the graph around the six attention
    # calls and around the unmask call; the K timed steps are K/M replays, and the
    # per-call times are those of the last replay's M steps, recorded inside the timed
    # region.
    M = max(d for d in range(1, min(10, args.steps) + 1) if args.steps % d == 0)
    ev = lambda: torch.cuda.Event(enable_timing=True, external=not args.no_graph)  # noqa: E731
    ev_attn = [(ev(), ev()) for _ in range(M if not args.no_graph else args.steps)]
    ev_unm = [(ev(), ev()) for _ in range(len(ev_attn))]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            wl.step(stream)
        stream.synchronize()
        graph = None
        if not args.no_graph:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for m in range(M):
                    wl.step(stream, ev_attn[m], ev_unm[m])
            graph.replay()  # one untimed replay
            stream.synchronize()
        # timed region: K steps with per-kernel events
        dist.barrier()
        torch.cuda.synchronize()
        clocks.mark_start()
        start.record(stream)
        if graph is not None:
            for _ in range(args.steps // M):
                graph.replay()
        else:
            for k in range(args.steps):
                wl.step(stream, ev_attn[k], ev_unm[k])
        end.record(stream)
        torch.cuda.synchronize()
        clocks.mark_end()
        dist.barrier()
    clk = clocks.stop()
    ms = start.elapsed_time(end) / args.steps
    ms_max = dist.max(ms)
    # the layers' calls run back to back between one event pair: the mean call time
    attn_ms = [s.elapsed_time(e) / len(wl.layers) for (s, e) in ev_attn]
    unm_ms = [s.elapsed_time(e) for (s, e) in ev_unm]
    attn_avg = float(np.mean(attn_ms))
    unm_avg = float(np.mean(unm_ms))
    peaks = measured_peaks()
    ab = wl.attn_bytes()
    achieved = ab / (attn_avg * 1e-3) / 1e9
    n = dist.world
    tokens_per_step = a.B * a.S * w.n_layers
    res = dict(
        metric=METRIC, value=n * tokens_per_step / (ms_max * 1e-3), unit=UNIT, n_gpus=n,
        steps=args.steps, warmup=args.warmup, ms_per_step=ms_max, higher_is_better=True,
        scaling="weak", vs_baseline=None, dtype="bf16",
        data="synthetic (seeded torch normals for Q/K/V, counter-generated logits)",
        config=dict(workload=w.name, B=a.B, S=a.S, Hq=a.Hq, Hkv=a.Hkv, d=a.d, Lmax=a.Lmax,
                    sum_ctx_len=int(wl.lens_np.sum()), V=w.V, attn_layers=w.n_layers,
                    temperature=w.temperature, gamma=w.threshold,
                    step="block_init + 6 x tt_block_attn (distinct layer K/V) + tt_confidence_unmask",
                    launch=("CUDA graph of %d steps replayed %d times; per-call times from the "
                            "events of the last replay (one pair around the 6 attention calls, "
                            "one around the unmask)" % (M, args.steps // M))
                    if not args.no_graph else "every kernel launched from the host",
                    l2="inputs larger than L2: 6 layer caches of %.0f MB visible K/V each" %
                       (ab / 1e6), parallelism=f"dp{n} (independent batches, no collective)"),
        roofline=dict(bound="hbm", achieved=achieved, peak=peaks["hbm_gbs"], unit="GB/s",
                      frac=achieved / peaks["hbm_gbs"], traffic=recorded_traffic(w.name),
                      kernel="tt_block_attn: block_attn_tc_kernel<128> + block_attn_merge_kernel<128>",
                      peak_source=peaks["source"],
                      algorithmic_bytes_per_launch=ab, avg_launch_ms=attn_avg),
        attn=dict(query_tokens_per_s=a.B * a.S / (attn_avg * 1e-3), hbm_gbs=achieved,
                  frac_of_measured=achieved / peaks["hbm_gbs"],
                  frac_of_8tbs=achieved / NORTH_STAR_HBM_GBS,
                  tflops=wl.attn_flops() / (attn_avg * 1e-3) / 1e12, avg_ms=attn_avg,
                  # the call is co-bound: against the bf16 tensor peak (sustained, since it
                  # is timed inside a long step), and the floor each roof sets for it
                  frac_of_bf16_sustained=wl.attn_flops() / (attn_avg * 1e-3) / 1e12 /
                  peaks["bf16_tflops_sustained"],
                  floor_ms_hbm=ab / peaks["hbm_gbs"] / 1e6,
                  floor_ms_tensor_sustained=wl.attn_flops() / peaks["bf16_tflops_sustained"] / 1e9),
        unmask=dict(positions_per_s=a.B * a.S / (unm_avg * 1e-3),
                    hbm_gbs=wl.unmask_bytes() / (unm_avg * 1e-3) / 1e9,
                    frac_of_measured=wl.unmask_bytes() / (unm_avg * 1e-3) / 1e9 / peaks["hbm_gbs"],
                    avg_ms=unm_avg),
        gpu_launches=wl.launches_per_step * args.steps,
        clocks=clk,
    )
    if not args.no_e2e:
        res["e2e"] = run_e2e(args, wl, stream, dist)
    del wl
    torch.cuda.empty_cache()
    return res


def run_e2e(args, wl: DeviceWorkload, stream, dist: Dist) -> dict:
    """Same step through the C ABI with host inputs: per step the block's Q/K/V of
    every layer, the logits and ctx_lens go host->device from pinned memory, and
    the step's result (tokens, commit flags, confidences) comes back.  The device
    inputs are double-buffered: a copy stream brings in step k+1's inputs while
    step k computes, as a serving loop would; every step still copies all of its
    inputs and reads back its result inside the timed region."""
    keys = ("q", "k_blk", "v_blk")
    # device input sets: set 0 = the workload's own tensors, set 1 = a second copy
    sets = [dict(layers=[{k: ly[k] for k in keys} for ly in wl.layers], logits=wl.logits,
                 lens=wl.lens)]
    sets.append(dict(layers=[{k: torch.empty_like(ly[k]) for k in keys} for ly in wl.layers],
                     logits=torch.empty_like(wl.logits), lens=torch.empty_like(wl.lens)))
    host_layers = [{k: ly[k].cpu().pin_memory() for k in keys} for ly in wl.layers]
    host_logits = wl.logits.cpu().pin_memory()
    host_lens = wl.lens.cpu().pin_memory()
    host_out = [(wl.tokens, torch.empty_like(wl.tokens, device="cpu").pin_memory()),
                (wl.masked, torch.empty_like(wl.masked, device="cpu").pin_memory()),
                (wl.conf, torch.empty_like(wl.conf, device="cpu").pin_memory())]
    h2d = (sum(h[k].numel() * h[k].element_size() for h in host_layers for k in keys) +
           host_logits.numel() * host_logits.element_size() +
           host_lens.numel() * host_lens.element_size())
    d2h = sum(h.numel() * h.element_size() for _, h in host_out)
    steps = max(3, min(args.steps, 20))
    copy_stream = torch.cuda.Stream()
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]

    def copy_in(i):
        st = sets[i]
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(done[i])  # the step that last read set i has finished
            for hl, dl in zip(host_layers, st["layers"]):
                for k in keys:
                    dl[k].copy_(hl[k], non_blocking=True)
            st["logits"].copy_(host_logits, non_blocking=True)
            st["lens"].copy_(host_lens, non_blocking=True)
            copied[i].record(copy_stream)

    def compute(i):
        st = sets[i]
        stream.wait_event(copied[i])
        for ly, dl in zip(wl.layers, st["layers"]):
            ly.update(dl)
        wl.logits, wl.lens = st["logits"], st["lens"]
        wl.step(stream)
        for d, h in host_out:
            h.copy_(d, non_blocking=True)
        done[i].record(stream)

    def run(n, start=None):
        if start is not None:
            copy_stream.wait_event(start)
        copy_in(0)
        for k in range(n):
            if k + 1 < n:
                copy_in((k + 1) % 2)
            compute(k % 2)

    with torch.cuda.stream(stream):
        for ev in done:
            ev.record(stream)
        run(2)
        torch.cuda.synchronize()
        dist.barrier()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        run(steps, start)
        end.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
    # restore the workload's own tensors
    for ly, dl in zip(wl.layers, sets[0]["layers"]):
        ly.update(dl)
    wl.logits, wl.lens = sets[0]["logits"], sets[0]["lens"]
    ms = dist.max(start.elapsed_time(end) / steps)
    a = wl.a
    return dict(value=dist.world * a.B * a.S * wl.w.n_layers / (ms * 1e-3), unit=UNIT,
                h2d_bytes_per_step=h2d, d2h_bytes_per_step=d2h, ms_per_step=ms, steps=steps,
                note="context K/V caches resident in HBM (the frozen tower's cache persists "
                     "across steps); per-step block inputs and logits copied from pinned host "
                     "memory on a copy stream, double-buffered so step k+1's copies overlap "
                     "step k's kernels; result copied back every step")


# ------------------------------------------------------------------ oracle (CPU) timing
def oracle_sample(w: synth.Workload, seqs, heads: int = 0, cache: Optional[dict] = None) -> dict:
    """Times the fp64 oracle on sequences `seqs` of the workload (one layer's attention,
    all heads, or the first `heads` query heads of one KV head's group, plus the unmask
    of the same rows).  Returns the query-token-layer units processed, the seconds an
    equivalent step share takes (attention + unmask/layers) and the threads used.  With a
    `cache` dict the generated inputs are kept and reused (only the oracle is timed)."""
    import oracle
    a = w.attn
    lens = synth.ctx_lens_for(a, w.seed)
    units, secs, threads = 0.0, 0.0, 0
    for b in seqs:
        L = int(lens[b])
        hkv, hq = (1, min(heads, a.Hq // a.Hkv)) if 0 < heads < a.Hq else (a.Hkv, a.Hq)
        key = (b, hq, hkv)
        if cache is not None and key in cache:
            inp = cache[key]
        else:
            shape = synth.AttnShape(1, a.S, hq, hkv, a.d, max(L, 1), lens=[L])
            inp = synth.attn_inputs(shape, seed=w.seed + 17 * b)
            if cache is not None:
                cache[key] = inp
        if cache is not None and "logits" in cache:
            logits = cache["logits"]
        else:
            logits = synth.counter_logits(w.seed, 0, 1, a.S, w.V, w.sigma, w.spike_p, "bf16")
            if cache is not None:
                cache["logits"] = logits
        t0 = time.perf_counter()
        _, _, used = oracle.block_attn(inp["q"], inp["k_ctx"], inp["v_ctx"], inp["ctx_lens"],
                                       inp["k_blk"], inp["v_blk"], return_threads=True)
        t1 = time.perf_counter()
        r = oracle.confidence_unmask(logits, "bf16", w.temperature, w.threshold, w.mask_token_id,
                                     np.full((1, a.S), w.mask_token_id, np.int32),
                                     np.ones((1, a.S), np.uint8))
        t2 = time.perf_counter()
        frac = hq / a.Hq
        units += a.S * frac
        secs += (t1 - t0) + (t2 - t1) * frac / w.n_layers
        threads = max(threads, used, r["threads"])
    return dict(units=units, secs=secs, threads=threads)


def cpu_baseline(w: synth.Workload, budget_s: float) -> dict:
    a = w.attn
    order = list(range(a.B))
    done, acc_units, acc_secs, threads = [], 0.0, 0.0, 0
    t_start = time.perf_counter()
    for b in order:
        r = oracle_sample(w, [b])
        done.append(b)
        acc_units += r["units"]
        acc_secs += r["secs"]
        threads = max(threads, r["threads"])
        if time.perf_counter() - t_start > budget_s:
            break
    lens = synth.ctx_lens_for(a, w.seed)
    return dict(value=acc_units / acc_secs, unit=UNIT, cores=threads, kind="oracle",
                sample=f"fp64 oracle, sequences {done} (ctx lens {[int(lens[b]) for b in done]}) "
                       f"of one attention layer, all heads, plus their unmask rows weighted 1/"
                       f"{w.n_layers}; {acc_secs:.1f} s of CPU work")


def run_reference(args, dist: Dist) -> dict:
    """The oracle as the reference arm: each step a bounded sample of the workload."""
    w = synth.workloads()[args.workload]
    a = w.attn
    budget = 240.0  # seconds of oracle work for the whole run
    cache: dict = {}
    n_samples = args.steps + max(0, args.warmup - 1)
    # Per step one sequence (cycling); as many query heads as fit the budget: all, one KV
    # head's group, then a half or a quarter of it, each candidate probed on the longest
    # sequence.  Fewer heads would leave the oracle timing mostly its K/V decode.
    G = a.Hq // a.Hkv
    longest = int(np.argmax(synth.ctx_lens_for(a, w.seed)))
    candidates = [a.Hq] + [G >> i for i in range(3) if (G >> i) >= 1]
    heads = candidates[-1]
    probe = None
    for h in candidates:
        probe = oracle_sample(w, [longest], h, cache)
        if probe["secs"] * n_samples <= budget:
            heads = h
            break
    units, secs, threads = 0.0, 0.0, probe["threads"]
    seq = 1
    for _ in range(max(0, args.warmup - 1)):
        oracle_sample(w, [seq % a.B], heads, cache)
        seq += 1
    for _ in range(args.steps):
        r = oracle_sample(w, [seq % a.B], heads, cache)
        seq += 1
        units += r["units"]
        secs += r["secs"]
        threads = max(threads, r["threads"])
    value = units / secs
    sample = ("fp64 oracle on the host cores; each step one sequence of the workload (cycling), "
              + ("all heads" if heads == a.Hq else f"{heads} query heads of one KV head's group")
              + f", one attention layer plus its unmask rows weighted 1/{w.n_layers}")
    return dict(
        impl="reference", metric=METRIC, value=value, unit=UNIT, n_gpus=dist.world,
        steps=args.steps, warmup=args.warmup, ms_per_step=1e3 * secs / max(args.steps, 1),
        higher_is_better=True, scaling="weak", vs_baseline=None, dtype="f64",
        data="synthetic (numpy PCG64 normals, counter-generated logits)",
        config=dict(workload=w.name, B=a.B, S=a.S, Hq=a.Hq, Hkv=a.Hkv, d=a.d, Lmax=a.Lmax,
                    V=w.V, attn_layers=w.n_layers),
        cpu_baseline=dict(kind="oracle", cores=threads, sample=sample, value=value, unit=UNIT),
        e2e=dict(value=value, unit=UNIT, h2d_bytes_per_step=0, d2h_bytes_per_step=0),
        gpu_launches=0)


def h2d_pinned_gbs(nbytes: int = 256 << 20, reps: int = 5) -> float:
    """Host-to-device copy rate from pinned memory (the link the e2e number crosses)."""
    host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dev = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    dev.copy_(host, non_blocking=True)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        dev.copy_(host, non_blocking=True)
    e1.record()
    torch.cuda.synchronize()
    return reps * nbytes / (e0.elapsed_time(e1) * 1e-3) / 1e9


def run_extras(args) -> dict:
    """Measurements of the other entry points, taken after the timed region (CUDA
    events around each call): the block loop over the sweep configuration (every S
    and gamma), block-by-block generation, Mamba-2 state seeding, the K/V append, and
    the host link's pinned copy rate."""
    from block_mask_diffusion_tt_b300 import profile
    ws = synth.workloads()
    w = ws[args.workload]
    peak = measured_peaks()["hbm_gbs"]
    out = {}
    sw = ws["sweep"]
    _, recs, _ = profile.run_loop(sw, 2, True)
    out["sweep"] = dict(workload=f"sweep B={sw.attn.B} V={sw.V} steps=S spike p 0.2->0.9 "
                                 f"T={sw.temperature}",
                        blocks=recs)
    _, gen, _ = profile.run_generate(w, 4, True)
    out["generate"] = dict(workload=w.name, max_new_tokens=4 * w.attn.S, **gen)
    us, gbs, how = profile.run_seed(w, 20, True)
    out["mamba_state_seed"] = dict(workload=f"{w.name} B={w.attn.B}, {how}", us=us, hbm_gbs=gbs,
                                   frac_of_measured=gbs / peak)
    us, gbs, how = profile.run_kvappend(w, 20, True)
    out["kv_append"] = dict(workload=f"{w.name}, {how}", us=us, hbm_gbs=gbs,
                            frac_of_measured=gbs / peak)
    out["h2d_pinned_gbs"] = h2d_pinned_gbs()
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="ragged16k", choices=sorted(synth.workloads()))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every kernel of every step from the host instead of replaying "
                         "a CUDA graph of the step")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the measurements of the other entry points (1 GPU only)")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    dist = Dist(args.gpus, init=args.impl == "ours")
    try:
        if args.impl == "reference":
            if dist.rank == 0:
                print(json.dumps(run_reference(args, dist)), flush=True)
            return
        res = run_ours(args, dist)
        if dist.world == 1 and not args.no_extras:
            res["extras"] = run_extras(args)
        if dist.rank == 0:
            if dist.world == 1:
                res["cpu_baseline"] = cpu_baseline(synth.workloads()[args.workload],
                                                   args.cpu_budget_s)
            print(json.dumps(res), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
