"""Seeded input generators: published test vectors, bf16 rounding, distribution checks."""
import numpy as np
import torch

from block_mask_diffusion_tt_b300 import synth


def test_splitmix64_published_sequence():
    # First outputs of the SplitMix64 reference generator seeded with 1234567.
    x, out = 1234567, []
    for _ in range(5):
        x = (x + synth.GAMMA) % (1 << 64)
        out.append(synth.mix64_int(x))
    assert out == [6457827717110365317, 3203168211198807973, 9817491932198370423,
                   4593380528125082431, 16408922859458223821]


def test_mix64_vectorised_matches_scalar():
    z = np.array([0, 1, 2**63, 2**64 - 1, 0x123456789ABCDEF0], dtype=np.uint64)
    assert [int(v) for v in synth.mix64(z)] == [synth.mix64_int(int(v)) for v in z]


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 7,
                        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.4e38, 1e-40],
                                 np.float32)])
    ours = synth.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(synth.bf16_to_f32(ours),
                          torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_counter_logits_distribution_and_determinism():
    z = synth.counter_logits(0, 3, 4, 16, 4096, 2.0, 0.0, dtype="f32")
    assert abs(z.mean()) < 0.02 and abs(z.std() - 2.0) < 0.02
    assert np.array_equal(z, synth.counter_logits(0, 3, 4, 16, 4096, 2.0, 0.0, dtype="f32"))
    assert not np.array_equal(z, synth.counter_logits(0, 4, 4, 16, 4096, 2.0, 0.0, dtype="f32"))
    # Irwin-Hall values are exact multiples of sigma/65536
    k = z.astype(np.float64) * 65536 / 2.0
    assert np.array_equal(k, np.round(k))


def test_counter_logits_spikes_and_row_subset():
    B, S, V = 8, 16, 512
    full = synth.counter_logits(1, 0, B, S, V, 2.0, 0.6, dtype="f32").reshape(B * S, V)
    has, tok = synth.spike_draws(1, 0, B * S, V, 0.6)
    assert 0.45 < has.mean() < 0.75
    base = synth.counter_logits(1, 0, B, S, V, 2.0, 0.0, dtype="f32").reshape(B * S, V)
    diff = full - base
    for r in range(B * S):
        nz = np.nonzero(diff[r])[0]
        assert (nz.tolist() == [tok[r]]) if has[r] else (len(nz) == 0)
    rows = np.array([5, 77, 3])
    sub = synth.counter_logits(1, 0, B, S, V, 2.0, 0.6, dtype="f32", rows=rows)
    assert np.array_equal(sub, full[rows])
    bits = synth.counter_logits(1, 0, B, S, V, 2.0, 0.6, dtype="bf16")
    assert np.array_equal(bits.reshape(B * S, V), synth.bf16_bits(full))


def test_spike_threshold_edges():
    assert synth.spike_threshold(0.0) == 0
    assert synth.spike_threshold(1.0) == 2**32
    has, _ = synth.spike_draws(0, 0, 1000, 10, 1.0)
    assert has.all()


def test_attn_inputs_shapes_and_lengths():
    w = synth.workloads()["ragged16k"]
    lens = synth.ctx_lens_for(w.attn, 0)
    assert lens.shape == (32,) and lens.min() >= 1024 and lens.max() <= 16384
    inp = synth.attn_inputs(synth.AttnShape(2, 4, 4, 2, 64, 10, lens=[3, 10]), 0, nan_pad=True)
    assert inp["q"].shape == (2, 4, 4, 64) and inp["k_ctx"].shape == (2, 2, 10, 64)
    assert np.isnan(synth.bf16_to_f32(inp["k_ctx"][0, :, 3:])).all()
    assert not np.isnan(synth.bf16_to_f32(inp["k_ctx"][0, :, :3])).any()
