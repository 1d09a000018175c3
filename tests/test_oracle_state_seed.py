"""Pins of the oracle's Mamba-2 state seeding (oracle.mamba_state_seed).

The expected destination is written out from a closed form: every source element
encodes (layer, part, sequence, position), so the seeded state must equal that code
for the sequences that take part, and the destination's own code elsewhere.  The
planted mistakes are those a seeding can make: the wrong layer, a sequence
swapped, the active mask ignored.
"""
import numpy as np
import pytest

import oracle

B, LAYERS = 5, 4
SHAPES = [(6, 3), (2, 4, 8)]  # per sequence: a conv state and an SSM state


def code(layer, part, b, shape, dst=False):
    pos = np.arange(int(np.prod(shape)), dtype=np.float64).reshape(shape)
    return (1e6 * (2 if dst else 1) + layer * 1e4 + part * 1e3 + b * 100 + pos).astype(np.float32)


def make(dst=False):
    return [[np.stack([code(l, p, b, s, dst) for b in range(B)]) for p, s in enumerate(SHAPES)]
            for l in range(LAYERS)]


@pytest.mark.parametrize("active", [None, np.array([1, 0, 1, 1, 0], np.uint8)])
def test_seed_equals_closed_form(active):
    out = oracle.mamba_state_seed(make(), make(dst=True), active)
    for l in range(LAYERS):
        for p, s in enumerate(SHAPES):
            for b in range(B):
                take = active is None or active[b]
                assert np.array_equal(out[l][p][b], code(l, p, b, s, dst=not take))


def _wrong_layer(src, dst, active=None):
    return oracle.mamba_state_seed(src[1:] + src[:1], dst, active)


def _swapped(src, dst, active=None):
    s2 = [[x[::-1].copy() for x in layer] for layer in src]
    return oracle.mamba_state_seed(s2, dst, active)


def _ignores_mask(src, dst, active=None):
    return oracle.mamba_state_seed(src, dst, None)


@pytest.mark.parametrize("mutant", [_wrong_layer, _swapped, _ignores_mask])
def test_planted_mistakes_fail_the_pin(mutant):
    active = np.array([1, 0, 1, 1, 0], np.uint8)
    out = mutant(make(), make(dst=True), active)
    ok = all(np.array_equal(out[l][p][b], code(l, p, b, s, dst=not active[b]))
             for l in range(LAYERS) for p, s in enumerate(SHAPES) for b in range(B))
    assert not ok
