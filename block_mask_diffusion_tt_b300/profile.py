"""Profiler driver: one operation of the denoiser step, called n times on a seeded
synthetic workload, so that a profiler can capture a single kernel launch on a
device footprint of one layer (a few hundred MB) rather than the whole step.

    python -m block_mask_diffusion_tt_b300.profile attn ragged16k 4
    python -m block_mask_diffusion_tt_b300.profile unmask ragged16k 4

`attn` runs `tt_block_attn` on one layer's block queries and context K/V;
`unmask` runs `tt_confidence_unmask` on a step where every position is masked.
"""
import argparse

import torch

from . import synth, tt


def run_attn(w: synth.Workload, n: int):
    a = w.attn
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed)

    def randn(shape):
        return torch.randn(shape, generator=g, device="cuda").to(torch.bfloat16)

    lens = torch.from_numpy(synth.ctx_lens_for(a, w.seed)).cuda()
    q = randn((a.B, a.S, a.Hq, a.d))
    k_ctx, v_ctx = randn((a.B, a.Hkv, a.Lmax, a.d)), randn((a.B, a.Hkv, a.Lmax, a.d))
    k_blk, v_blk = randn((a.B, a.S, a.Hkv, a.d)), randn((a.B, a.S, a.Hkv, a.d))
    out = torch.empty_like(q)
    ws = tt.Workspace(tt.block_attn_workspace_size(tt.attn_desc(q, k_ctx, v_ctx, k_blk, v_blk,
                                                                 out)))
    for _ in range(n):
        tt.block_attn(q, k_ctx, v_ctx, lens, k_blk, v_blk, out=out, workspace=ws)


def run_unmask(w: synth.Workload, n: int):
    a = w.attn
    logits = tt.synth_logits(w.seed, 0, a.B, a.S, w.V, w.sigma,
                             synth.spike_threshold(w.spike_p), tt.TT_BF16)
    tokens = torch.empty((a.B, a.S), dtype=torch.int32, device="cuda")
    masked = torch.empty((a.B, a.S), dtype=torch.uint8, device="cuda")
    for _ in range(n):
        tt.block_init(tokens, masked, w.mask_token_id)
        tt.confidence_unmask(logits, tokens, masked, w.temperature, w.threshold,
                             w.mask_token_id)


def main():
    ap = argparse.ArgumentParser(description="run one op of the step n times")
    ap.add_argument("op", choices=["attn", "unmask"])
    ap.add_argument("workload", choices=sorted(synth.workloads()))
    ap.add_argument("n", type=int, nargs="?", default=4)
    args = ap.parse_args()
    tt.load()
    w = synth.workloads()[args.workload]
    (run_attn if args.op == "attn" else run_unmask)(w, args.n)
    torch.cuda.synchronize()
    print("ok", args.op, w.name, args.n)


if __name__ == "__main__":
    main()
