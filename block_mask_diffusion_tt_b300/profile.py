"""Profiler driver: one operation of the denoiser step, called n times on a seeded
synthetic workload, so that a profiler can capture a single kernel launch on a
device footprint of one layer (a few hundred MB) rather than the whole step.

    python -m block_mask_diffusion_tt_b300.profile attn ragged16k 4
    python -m block_mask_diffusion_tt_b300.profile unmask ragged16k 4

`attn` runs `tt_block_attn` on one layer's block queries and context K/V;
`unmask` runs `tt_confidence_unmask` on a step where every position is masked;
`loop` runs `tt_denoise_block_loop` with the library's synthetic logits producer
over the sweep configuration's block sizes and thresholds (steps = S), and reports
committed tokens/s and the steps used per block;
`kvappend` runs `tt_kv_append` for every attention layer of the workload (a
committed block of S rows joins each layer's context cache);
`seed` runs `tt_mamba_state_seed` over 23 Mamba-2 layers for the workload's batch;
`generate` runs `tt_generate_blocks` for n blocks of the workload.

With --time it instead times back-to-back calls with CUDA events and prints the
mean time per call and the algorithmic bandwidth.  The timed calls go to the C ABI
with arguments built once, so host work does not leave the GPU idle between
kernels.  For attention it cycles over enough layers (each with its own K/V) that
their caches together exceed twice the L2 size, so no call finds its K/V in L2.
"""
import argparse
import ctypes

import numpy as np
import torch

from . import synth, tt

L2_BYTES = 126 * 1024 * 1024


def _attn_layer(a, g):
    def randn(shape):
        return torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)

    q = randn((a.B, a.S, a.Hq, a.d))
    return dict(q=q, k_ctx=randn((a.B, a.Hkv, a.Lmax, a.d)), v_ctx=randn((a.B, a.Hkv, a.Lmax, a.d)),
                k_blk=randn((a.B, a.S, a.Hkv, a.d)), v_blk=randn((a.B, a.S, a.Hkv, a.d)),
                out=torch.empty_like(q))


def attn_bytes(a, lens_np) -> int:
    """Algorithmic bytes of one call: visible K/V, block K/V, Q and O (bf16)."""
    kv = int(lens_np.astype(np.int64).sum()) * a.Hkv * a.d * 2 * 2
    return kv + a.B * a.S * a.Hkv * a.d * 2 * 2 + a.B * a.S * a.Hq * a.d * 2 * 2


def _graph_us(fn, n: int) -> float:
    """Device time per call of fn(i) for i < n: the n calls are captured in one CUDA
    graph and its replay is timed with CUDA events, so the host's launch cost does
    not enter (a small call enqueues in about as long as it runs)."""
    fn(0)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for i in range(n):
            fn(i)
    graph.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / n


def run_attn(w: synth.Workload, n: int, time_it: bool = False, graph: bool = False):
    a = w.attn
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed)
    lens_np = synth.ctx_lens_for(a, w.seed)
    lens = torch.from_numpy(lens_np).cuda()
    cache = a.B * a.Hkv * a.Lmax * a.d * 2 * 2
    nl = max(2, -(-2 * L2_BYTES // cache)) if time_it else 1
    layers = [_attn_layer(a, g) for _ in range(nl)]
    l0 = layers[0]
    ws = tt.Workspace(tt.block_attn_workspace_size(
        tt.attn_desc(l0["q"], l0["k_ctx"], l0["v_ctx"], l0["k_blk"], l0["v_blk"], l0["out"])))

    if not time_it:
        for _ in range(n):
            tt.block_attn(l0["q"], l0["k_ctx"], l0["v_ctx"], lens, l0["k_blk"], l0["v_blk"],
                          out=l0["out"], workspace=ws)
        return None
    lib = tt.load()
    desc = tt.attn_desc(l0["q"], l0["k_ctx"], l0["v_ctx"], l0["k_blk"], l0["v_blk"], l0["out"])
    sp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    argv = [(ctypes.byref(desc), tt._ptr(ly["q"]), tt._ptr(ly["k_ctx"]), tt._ptr(ly["v_ctx"]),
             tt._ptr(lens), tt._ptr(ly["k_blk"]), tt._ptr(ly["v_blk"]), tt._ptr(ly["out"]), None,
             ws.ptr, ws.nbytes, sp) for ly in layers]

    def call(i):
        tt.check(lib.tt_block_attn(*argv[i]))

    if graph:
        def gcall(i):  # on the stream being captured
            cs = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            tt.check(lib.tt_block_attn(*(argv[i % nl][:-1] + (cs,))))

        us = _graph_us(gcall, max(n, nl))
        return us, attn_bytes(a, lens_np) / us / 1e3, f"{nl} layers, one CUDA graph"
    for _ in range(3):
        for i in range(nl):
            call(i)
    torch.cuda.synchronize()
    rounds = max(1, -(-n // nl))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(rounds):
        for i in range(nl):
            call(i)
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (rounds * nl)
    return us, attn_bytes(a, lens_np) / us / 1e3, f"{nl} layers"


def run_unmask(w: synth.Workload, n: int, time_it: bool = False, graph: bool = False):
    a = w.attn
    logits = tt.synth_logits(w.seed, 0, a.B, a.S, w.V, w.sigma,
                             synth.spike_threshold(w.spike_p), tt.TT_BF16)
    tokens = torch.empty((a.B, a.S), dtype=torch.int32, device="cuda")
    masked = torch.empty((a.B, a.S), dtype=torch.uint8, device="cuda")
    desc = tt.unmask_desc(a.B, a.S, w.V, tt.TT_BF16, w.temperature, w.threshold, w.mask_token_id)
    ws = tt.Workspace(tt.confidence_unmask_workspace_size(desc))
    if not time_it:
        for _ in range(n):
            tt.block_init(tokens, masked, w.mask_token_id)
            tt.confidence_unmask(logits, tokens, masked, w.temperature, w.threshold,
                                 w.mask_token_id, workspace=ws)
        return None
    lib = tt.load()
    sp = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    conf = torch.empty((a.B, a.S), dtype=torch.float32, device="cuda")
    now = torch.empty((a.B, a.S), dtype=torch.uint8, device="cuda")
    remaining = torch.empty((a.B,), dtype=torch.int32, device="cuda")
    init_args = (ctypes.byref(desc), tt._ptr(tokens), tt._ptr(masked), None, None, sp)
    unmask_args = (ctypes.byref(desc), tt._ptr(logits), tt._ptr(tokens), tt._ptr(masked),
                   tt._ptr(conf), tt._ptr(now), tt._ptr(remaining), 0, ws.ptr, ws.nbytes, sp)
    nbytes = a.B * a.S * w.V * 2 + a.B * a.S * (4 + 1 + 4 + 1 + 4) + a.B * 4
    if graph:
        def both(i):
            cs = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            tt.check(lib.tt_block_init(*(init_args[:-1] + (cs,))))
            tt.check(lib.tt_confidence_unmask(*(unmask_args[:-1] + (cs,))))

        def init_only(i):
            cs = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            tt.check(lib.tt_block_init(*(init_args[:-1] + (cs,))))

        us = _graph_us(both, n) - _graph_us(init_only, n)
        return us, nbytes / us / 1e3, "one CUDA graph, block init subtracted"
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for i in range(3 + n):
        tt.check(lib.tt_block_init(*init_args))
        if i >= 3:
            ev[i - 3][0].record()
        tt.check(lib.tt_confidence_unmask(*unmask_args))
        if i >= 3:
            ev[i - 3][1].record()
    torch.cuda.synchronize()
    us = sum(s.elapsed_time(e) for s, e in ev) * 1e3 / n
    # every position is masked at a block's first step: whole rows plus the state arrays
    return us, nbytes / us / 1e3, "events around each call"


def run_loop(w: synth.Workload, n: int, time_it: bool = False):
    """One block per (S, gamma) of the workload's sweep (or its own S and gamma),
    n times each; with time_it, the mean time of a block and what it committed (as
    text lines and as one record per (S, gamma))."""
    a = w.attn
    ex = w.extra or {}
    s_values = ex.get("S_values", (a.S,))
    gammas = ex.get("gammas", (w.threshold,))
    lines, records = [], []
    for S in s_values:
        ps = [synth.sweep_spike_p(k, S, ex.get("spike_p_first", w.spike_p),
                                  ex.get("spike_p_last", w.spike_p)) for k in range(S)]
        params = tt.synth_params(w.seed, a.B, S, w.V, tt.TT_BF16, w.sigma,
                                 [synth.spike_threshold(p) for p in ps])
        logits = torch.empty((a.B, S, w.V), dtype=torch.bfloat16, device="cuda")
        tokens = torch.empty((a.B, S), dtype=torch.int32, device="cuda")
        masked = torch.empty((a.B, S), dtype=torch.uint8, device="cuda")
        used = torch.empty((a.B,), dtype=torch.int32, device="cuda")
        desc = tt.unmask_desc(a.B, S, w.V, tt.TT_BF16, w.temperature, 0.5, w.mask_token_id)
        ws = tt.Workspace(tt.denoise_block_loop_workspace_size(desc))
        for gamma in gammas:
            def block():
                return tt.denoise_block_loop(a.B, S, w.V, tt.TT_BF16, w.temperature, gamma,
                                             w.mask_token_id, S, tokens, masked, used,
                                             logits_buf=logits, synth=params, workspace=ws)
            block()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(n):
                steps = block()
            e1.record()
            torch.cuda.synchronize()
            if time_it:
                us = e0.elapsed_time(e1) * 1e3 / n
                mean_used = float(used.float().mean())
                lines.append(f"S={S:2d} gamma={gamma:.2f}: {us:8.1f} us per block, "
                             f"{a.B * S / us * 1e6:12.0f} committed tokens/s, "
                             f"steps used per block {mean_used:.2f} (loop ran {steps})")
                records.append(dict(S=S, gamma=gamma, us_per_block=us,
                                    committed_tokens_per_s=a.B * S / us * 1e6,
                                    steps_per_block=mean_used,
                                    max_steps_per_block=int(used.max())))
    return ("\n".join(lines), records, None) if time_it else None


def run_kvappend(w: synth.Workload, n: int, time_it: bool = False):
    """tt_kv_append of one committed block into every attention layer of the workload.

    With time_it, n appends are captured in a CUDA graph and the replay is timed with
    CUDA events: a call enqueues in more time than the kernel takes, so timing the
    calls from the host would measure the host.  Each append lands S rows further on
    (the lengths start low enough for all n), so every call moves the same bytes."""
    a = w.attn
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed)

    def randn(shape):
        return torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)

    L = w.n_layers
    kc = [randn((a.B, a.Hkv, a.Lmax, a.d)) for _ in range(L)]
    vc = [randn((a.B, a.Hkv, a.Lmax, a.d)) for _ in range(L)]
    kb = [randn((a.B, a.S, a.Hkv, a.d)) for _ in range(L)]
    vb = [randn((a.B, a.S, a.Hkv, a.d)) for _ in range(L)]
    room = a.Lmax - (n + 1) * a.S
    if room < 0:
        raise ValueError(f"Lmax={a.Lmax} has no room for {n} appends of {a.S} rows")
    lens0 = torch.from_numpy(np.minimum(synth.ctx_lens_for(a, w.seed), room)).cuda()
    lens = lens0.clone()
    if not time_it:
        for _ in range(n):
            tt.kv_append(kc, vc, lens, kb, vb)
        return None
    tt.kv_append(kc, vc, lens, kb, vb)  # warm-up outside the graph
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(n):
            tt.kv_append(kc, vc, lens, kb, vb)
    lens.copy_(lens0)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    graph.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / n
    moved = int((lens - lens0).min().item())
    assert moved == n * a.S, f"appends in the graph moved lengths by {moved}"
    nbytes = 2 * (L * 2 * a.B * a.S * a.Hkv * a.d * 2)  # each block row read once, written once
    return us, nbytes / us / 1e3, f"{L} layers, {n} calls in one CUDA graph"


# Mamba-2 layer shapes used for the seeding measurement: 23 layers (the pages' count);
# per layer and sequence a conv state of 6144 channels x 3 taps in bf16 and an SSM
# state of 64 heads x 64 x 128 in fp32 (a Mamba-2 layer with 64 heads of 64, state
# size 128, 8 groups, conv width 4 -- the pages give no layer dimensions).
SEED_LAYERS = 23
SEED_CONV = (6144, 3)
SEED_SSM = (64, 64, 128)


def run_seed(w: synth.Workload, n: int, time_it: bool = False):
    """tt_mamba_state_seed of every Mamba-2 layer for the workload's batch; with time_it,
    n calls captured in a CUDA graph and the replay timed (bytes read + written)."""
    B = w.attn.B
    src = [[torch.randn((B,) + SEED_CONV, device="cuda").to(torch.bfloat16),
            torch.randn((B,) + SEED_SSM, device="cuda")] for _ in range(SEED_LAYERS)]
    dst = [[torch.empty_like(a) for a in layer] for layer in src]
    if not time_it:
        for _ in range(n):
            tt.mamba_state_seed(src, dst)
        return None
    tt.mamba_state_seed(src, dst)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(n):
            tt.mamba_state_seed(src, dst)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    graph.replay()
    e1.record()
    torch.cuda.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / n
    per_seq = sum(a[0].numel() * a.element_size() for a in src[0])
    nbytes = 2 * SEED_LAYERS * B * per_seq
    return us, nbytes / us / 1e3, f"{SEED_LAYERS} layers, {n} calls in one CUDA graph"


def run_generate(w: synth.Workload, n: int, time_it: bool = False):
    """tt_generate_blocks on the workload's batch: n blocks of S positions, logits from
    the counter generator per (block, step), synthetic K/V appended to the workload's
    attention layers; with time_it, generated tokens per second over the whole call."""
    a = w.attn
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed)
    L = w.n_layers
    Lmax = a.Lmax + n * a.S
    kc = [torch.randn((a.B, a.Hkv, Lmax, a.d), generator=g, device="cuda").to(torch.bfloat16)
          for _ in range(L)]
    vc = [torch.randn((a.B, a.Hkv, Lmax, a.d), generator=g, device="cuda").to(torch.bfloat16)
          for _ in range(L)]
    kb = [torch.empty((a.B, a.S, a.Hkv, a.d), dtype=torch.bfloat16, device="cuda")
          for _ in range(L)]
    vb = [torch.empty_like(x) for x in kb]
    lens = torch.from_numpy(synth.ctx_lens_for(a, w.seed)).cuda()
    thr = synth.spike_threshold(w.spike_p)

    def logits_fn(block, step, buf):
        tt.synth_logits(w.seed + block, step, a.B, a.S, w.V, w.sigma, thr, tt.TT_BF16, out=buf)

    def kv_fn(block, tokens, active, k_blk, v_blk):
        for layer in range(L):
            tt.synth_logits(1000 + block * L + layer, 0, a.B, a.S, a.Hkv * a.d, 1.0, 0,
                            tt.TT_BF16, out=k_blk[layer].view(a.B, a.S, a.Hkv * a.d))
            tt.synth_logits(2000 + block * L + layer, 0, a.B, a.S, a.Hkv * a.d, 1.0, 0,
                            tt.TT_BF16, out=v_blk[layer].view(a.B, a.S, a.Hkv * a.d))

    max_new = n * a.S
    out = torch.empty((a.B, max_new), dtype=torch.int32, device="cuda")
    gen_len = torch.zeros((a.B,), dtype=torch.int32, device="cuda")
    active = torch.ones((a.B,), dtype=torch.uint8, device="cuda")
    steps = torch.zeros((a.B,), dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    blocks = tt.generate_blocks(logits_fn, kv_fn, w.V, tt.TT_BF16, w.temperature, w.threshold,
                                w.mask_token_id, w.steps_per_block, max_new, -1, kc, vc, lens,
                                kb, vb, out, gen_len, active, steps)
    e1.record()
    torch.cuda.synchronize()
    if not time_it:
        return None
    us = e0.elapsed_time(e1) * 1e3
    toks = int(gen_len.sum())
    mean_steps = float(steps.float().mean()) / max(blocks, 1)
    return (f"{blocks} blocks, {toks} tokens in {us / 1e3:.2f} ms: {toks / us * 1e6:.0f} "
            f"generated tokens/s, {mean_steps:.2f} steps per block",
            dict(blocks=blocks, tokens=toks, ms=us / 1e3, generated_tokens_per_s=toks / us * 1e6,
                 steps_per_block=mean_steps), None)


def main():
    ap = argparse.ArgumentParser(description="run one op of the step n times")
    ap.add_argument("op", choices=["attn", "unmask", "loop", "kvappend", "seed", "generate"])
    ap.add_argument("workload", choices=sorted(synth.workloads()))
    ap.add_argument("n", type=int, nargs="?", default=4)
    ap.add_argument("--time", action="store_true",
                    help="time n back-to-back calls with CUDA events instead")
    ap.add_argument("--graph", action="store_true",
                    help="with --time (attn, unmask): time a CUDA-graph replay of the n calls")
    args = ap.parse_args()
    tt.load()
    w = synth.workloads()[args.workload]
    run = dict(attn=run_attn, unmask=run_unmask, loop=run_loop, kvappend=run_kvappend,
               seed=run_seed, generate=run_generate)[args.op]
    res = run(w, args.n, args.time, args.graph) if args.op in ("attn", "unmask") else \
        run(w, args.n, args.time)
    torch.cuda.synchronize()
    if res is None:
        print("ok", args.op, w.name, args.n)
    elif args.op in ("loop", "generate"):
        print(f"{args.op} {w.name}:\n{res[0]}")
    else:
        us, gbs, how = res
        print(f"{args.op} {w.name}: {us:.1f} us per call, {gbs:.0f} GB/s ({how})")


if __name__ == "__main__":
    main()
