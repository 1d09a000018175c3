"""The multi-rank path of bench.py on CPU: two processes over the gloo backend.

bench.py runs one process per GPU.  Ranks take independent batches and exchange no
data; the only collectives are the barriers around the timed region and the
max-over-ranks of the step time.  These tests run that plumbing with world size 2
on the host, and launch the reference arm the way the N>1 bench is launched
(torch.distributed.run), where rank 0 alone prints the result line.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_RANK_CODE = r"""
import json, os, sys
sys.path.insert(0, os.environ["TT_ROOT"])
import bench
from block_mask_diffusion_tt_b300 import synth
world, rank = int(os.environ["WORLD_SIZE"]), int(os.environ["RANK"])
d = bench.Dist(world)
try:
    assert d.pg is not None, "no process group"
    d.barrier()
    # per-rank step times: the job's time is the slowest rank's
    got = d.max(1.5 * (rank + 1))
    d.barrier()
    w = synth.workloads()["ragged16k"]
    lens = synth.ctx_lens_for(w.attn, bench.rank_seed(w, rank)).tolist()
    print(json.dumps(dict(rank=rank, max=got, lens=lens)), flush=True)
finally:
    d.close()
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(**kw) -> dict:
    env = dict(os.environ)
    env.update({k: str(v) for k, v in kw.items()})
    env.update(TT_ROOT=ROOT, CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="2")
    return env


def test_two_gloo_ranks_max_barrier_and_independent_batches():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", _RANK_CODE], cwd=ROOT,
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                              env=_env(MASTER_ADDR="127.0.0.1", MASTER_PORT=port, WORLD_SIZE=2,
                                       RANK=r, LOCAL_RANK=r))
             for r in range(2)]
    outs = []
    try:
        for p in procs:
            out, err = p.communicate(timeout=240)
            assert p.returncode == 0, err[-2000:]
            outs.append(json.loads(out.strip().splitlines()[-1]))
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    by_rank = {o["rank"]: o for o in outs}
    assert sorted(by_rank) == [0, 1]
    # the max over ranks reaches every rank
    assert by_rank[0]["max"] == by_rank[1]["max"] == 3.0
    # each rank draws its own batch (weak scaling): the context lengths differ
    assert by_rank[0]["lens"] != by_rank[1]["lens"]
    assert all(1024 <= L <= 16384 for o in outs for L in o["lens"])


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3",
           "--workload", "tiny"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=_env())
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip().startswith("{")]
    assert len(lines) == 1, r.stdout
    res = json.loads(lines[0])
    assert res["impl"] == "reference"
    assert res["n_gpus"] == 2 and res["steps"] == 1 and res["warmup"] == 3
    assert res["value"] > 0 and np.isfinite(res["value"])
    assert res["e2e"]["h2d_bytes_per_step"] == 0 and res["e2e"]["d2h_bytes_per_step"] == 0
    assert res["cpu_baseline"]["kind"] == "oracle" and res["cpu_baseline"]["cores"] >= 1
