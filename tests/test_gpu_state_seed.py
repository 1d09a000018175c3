"""GPU parity of tt_mamba_state_seed: byte work, compared bit for bit with the oracle,
including every state the seeding must leave untouched."""
import numpy as np
import pytest
import torch

import oracle
from block_mask_diffusion_tt_b300 import tt
import _gpu

pytestmark = pytest.mark.gpu


def _rand(rng, shape, dtype):
    n = int(np.prod(shape)) * np.dtype(dtype).itemsize
    return rng.integers(0, 256, size=n, dtype=np.uint8).view(dtype).reshape(shape)


def _to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.uint8)).to(_gpu.DEV).view(
        {np.uint16: torch.bfloat16, np.float32: torch.float32}[a.dtype.type]).view(a.shape)


def _back(t, dtype):
    """The tensor's bytes as `dtype` values (compared through their bit patterns)."""
    return t.contiguous().view(torch.uint8).cpu().numpy().view(dtype).reshape(tuple(t.shape))


def _same(a, b):
    return np.array_equal(np.ascontiguousarray(a).view(np.uint8), np.ascontiguousarray(b).view(np.uint8))


@pytest.mark.parametrize("B,layers,active", [
    (5, 23, [1, 0, 1, 1, 0]),   # the pages' 23 Mamba-2 layers
    (3, 1, None),
    (40, 4, None),
])
def test_seed_matches_oracle(B, layers, active):
    rng = np.random.default_rng(B * 100 + layers)
    shapes = [((B, 768, 3), np.uint16), ((B, 8, 64, 32), np.float32)]  # conv (bf16), SSM (fp32)
    src = [[_rand(rng, s, t) for s, t in shapes] for _ in range(layers)]
    dst = [[_rand(rng, s, t) for s, t in shapes] for _ in range(layers)]
    act = None if active is None else np.asarray(active, np.uint8)
    ref = oracle.mamba_state_seed(src, dst, act)
    dsrc = [[_to_dev(x) for x in layer] for layer in src]
    ddst = [[_to_dev(x) for x in layer] for layer in dst]
    tt.mamba_state_seed(dsrc, ddst, None if act is None else torch.from_numpy(act).to(_gpu.DEV))
    torch.cuda.synchronize()
    for l in range(layers):
        for p, (_, t) in enumerate(shapes):
            assert _same(_back(ddst[l][p], t), ref[l][p]), (l, p)


def test_seed_into_strided_destination():
    """Destination states that sit inside larger per-sequence buffers (stride > size):
    the bytes between them are not touched."""
    rng = np.random.default_rng(3)
    B, layers = 4, 3
    src = [[_rand(rng, (B, 16, 32), np.float32)] for _ in range(layers)]
    big = [_rand(rng, (B, 20, 32), np.float32) for _ in range(layers)]
    dbig = [_to_dev(x) for x in big]
    tt.mamba_state_seed([[_to_dev(x[0])] for x in src], [[t[:, :16]] for t in dbig])
    torch.cuda.synchronize()
    for l in range(layers):
        got = _back(dbig[l], np.float32)
        assert _same(got[:, :16], src[l][0])
        assert _same(got[:, 16:], big[l][:, 16:])
