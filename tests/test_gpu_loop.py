"""GPU parity of tt_denoise_block_loop and of the device synthetic-logits generator."""
import numpy as np
import pytest
import torch

import oracle
from block_mask_diffusion_tt_b300 import synth, tt
import _gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,sigma,p", [("bf16", 2.0, 0.6), ("f32", 3.0, 0.0), ("bf16", 1.0, 1.0)])
def test_device_generator_matches_python(dtype, sigma, p):
    B, S, V = 3, 16, 4099
    for step in (0, 5):
        ref = synth.counter_logits(42, step, B, S, V, sigma, p, dtype)
        got = tt.synth_logits(42, step, B, S, V, sigma, synth.spike_threshold(p),
                              tt.TT_BF16 if dtype == "bf16" else tt.TT_F32)
        torch.cuda.synchronize()
        g = got.view(torch.int16).cpu().numpy().view(np.uint16) if dtype == "bf16" else \
            got.cpu().numpy()
        assert np.array_equal(g, ref)


def _state(B, S):
    return (torch.zeros((B, S), dtype=torch.int32, device=_gpu.DEV),
            torch.zeros((B, S), dtype=torch.uint8, device=_gpu.DEV),
            torch.zeros((B,), dtype=torch.int32, device=_gpu.DEV),
            torch.zeros((B, S), dtype=torch.int32, device=_gpu.DEV))


def _compare(ref, tokens, masked, steps_used, cstep, b_slice=slice(None)):
    assert ref["ambiguous"] == 0
    assert np.array_equal(tokens.cpu().numpy()[b_slice], ref["tokens"])
    assert np.array_equal(masked.cpu().numpy()[b_slice], ref["is_masked"])
    assert np.array_equal(steps_used.cpu().numpy()[b_slice], ref["steps_used"])
    assert np.array_equal(cstep.cpu().numpy()[b_slice], ref["committed_step"])


def test_tiny_config_loop_with_device_producer():
    w = synth.workloads()["tiny"]
    B, S, V = w.attn.B, w.attn.S, w.V
    ref = oracle.block_loop(B, S, lambda k: synth.counter_logits(w.seed, k, B, S, V, w.sigma, 0.0,
                                                                  "f32"),
                            "f32", w.temperature, w.threshold, w.mask_token_id, w.steps_per_block)
    tokens, masked, steps_used, cstep = _state(B, S)
    params = tt.synth_params(w.seed, B, S, V, tt.TT_F32, w.sigma, [0])
    n = tt.denoise_block_loop(B, S, V, tt.TT_F32, w.temperature, w.threshold, w.mask_token_id,
                              w.steps_per_block, tokens, masked, steps_used, cstep, synth=params)
    torch.cuda.synchronize()
    _compare(ref, tokens, masked, steps_used, cstep)
    assert n == int(ref["steps_used"].max())
    assert not masked.any()


def test_loop_with_python_producer_and_resume():
    B, S, V = 3, 16, 700
    fn = lambda k: synth.counter_logits(1, k, B, S, V, 0.25, 0.15, "f32")  # noqa: E731
    ref = oracle.block_loop(B, S, fn, "f32", 0.1, 0.95, 3, 16)

    def producer(step, buf):
        buf.copy_(torch.from_numpy(fn(step)).to(buf.device), non_blocking=False)

    tokens, masked, steps_used, cstep = _state(B, S)
    n1 = tt.denoise_block_loop(B, S, V, tt.TT_F32, 0.1, 0.95, 3, 16, tokens, masked, steps_used,
                               cstep, producer=producer, stop_step=8)
    assert n1 == 8 and masked.any()
    n2 = tt.denoise_block_loop(B, S, V, tt.TT_F32, 0.1, 0.95, 3, 16, tokens, masked, steps_used,
                               cstep, producer=producer, start_step=8)
    torch.cuda.synchronize()
    _compare(ref, tokens, masked, steps_used, cstep)
    assert n1 + n2 == int(ref["steps_used"].max())


@pytest.mark.parametrize("gamma,steps", [(0.0, 16), (1.5, 16), (1.5, 5), (0.8, 16)])
def test_loop_thresholds_and_forced_last_step(gamma, steps):
    B, S, V = 4, 16, 2048
    thr = [synth.spike_threshold(0.3)]
    fn = lambda k: synth.counter_logits(3, k, B, S, V, 1.0, 0.3, "bf16")  # noqa: E731
    ref = oracle.block_loop(B, S, fn, "bf16", 0.1, gamma, 3, steps)
    tokens, masked, steps_used, cstep = _state(B, S)
    tt.denoise_block_loop(B, S, V, tt.TT_BF16, 0.1, gamma, 3, steps, tokens, masked, steps_used,
                          cstep, synth=tt.synth_params(3, B, S, V, tt.TT_BF16, 1.0, thr))
    torch.cuda.synchronize()
    _compare(ref, tokens, masked, steps_used, cstep)
    if gamma == 0.0:
        assert (steps_used.cpu().numpy() == 1).all()
    if gamma > 1.0:
        assert (steps_used.cpu().numpy() == min(S, steps)).all()


def test_sweep_config_sampled_sequences():
    """Sweep shape at S=16, gamma=0.8: full batch on the GPU, first two sequences in the oracle."""
    w = synth.workloads()["sweep"]
    B, S, V = w.attn.B, 16, w.V
    ps = [synth.sweep_spike_p(k, S) for k in range(S)]
    tokens, masked, steps_used, cstep = _state(B, S)
    tt.denoise_block_loop(B, S, V, tt.TT_BF16, 0.1, 0.8, 3, S, tokens, masked, steps_used, cstep,
                          synth=tt.synth_params(w.seed, B, S, V, tt.TT_BF16, w.sigma,
                                                _gpu.synth_thresholds(ps)))
    torch.cuda.synchronize()
    Bs = 2  # rows b*S+s of the first sequences are the same draws in a smaller batch
    ref = oracle.block_loop(Bs, S, lambda k: synth.counter_logits(w.seed, k, Bs, S, V, w.sigma,
                                                                   ps[k], "bf16"),
                            "bf16", 0.1, 0.8, 3, S)
    _compare(ref, tokens, masked, steps_used, cstep, slice(0, Bs))


def test_producer_error_stops_loop():
    B, S, V = 2, 8, 100
    tokens, masked, steps_used, cstep = _state(B, S)

    def producer(step, buf):
        if step == 2:
            raise RuntimeError("planted producer failure")
        buf.copy_(torch.from_numpy(synth.counter_logits(0, step, B, S, V, 0.25, 0.0, "f32"))
                  .to(buf.device))

    with pytest.raises(tt.TTError) as e:
        tt.denoise_block_loop(B, S, V, tt.TT_F32, 0.1, 1.5, 3, 8, tokens, masked, steps_used,
                              cstep, producer=producer)
    assert e.value.status == tt.TT_ERR_CALLBACK
    torch.cuda.synchronize()
    assert (steps_used.cpu().numpy() == 2).all()  # two finished steps, state consistent
    assert (masked.cpu().numpy().sum(axis=1) == S - 2).all()


def test_host_watchdog_reports_timeout_and_state_stays_resumable():
    """The loop's bounded host wait: a producer whose stream work is held up on the
    host (a host function that sleeps 300 ms, enqueued through the driver API) makes
    the per-step wait run out after timeout_ms = 50.  The call returns TT_ERR_TIMEOUT
    having counted no finished step; once the stream drains, the device state is that
    of step 0, and a resumed call finishes the block exactly as the oracle does."""
    import ctypes
    import time

    B, S, V = 2, 8, 300
    fn = lambda k: synth.counter_logits(4, k, B, S, V, 0.25, 0.2, "f32")  # noqa: E731
    cuda = ctypes.CDLL("libcuda.so.1")
    cuda.cuLaunchHostFunc.restype = ctypes.c_int
    cuda.cuLaunchHostFunc.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    HOSTFN = ctypes.CFUNCTYPE(None, ctypes.c_void_p)
    slept = []

    def _sleep(_user):
        time.sleep(0.3)
        slept.append(1)

    host_fn = HOSTFN(_sleep)
    # logits staged on the device first: a copy from pageable host memory would wait
    # for the stream (and so for the sleeping host function) before the loop's wait
    staged = [torch.from_numpy(fn(k)).to(_gpu.DEV) for k in range(S)]
    torch.cuda.synchronize()

    def producer(step, buf):
        if step == 0:
            s = torch.cuda.current_stream().cuda_stream
            assert cuda.cuLaunchHostFunc(ctypes.c_void_p(s), ctypes.cast(host_fn, ctypes.c_void_p),
                                         None) == 0
        buf.copy_(staged[step], non_blocking=True)

    tokens, masked, steps_used, cstep = _state(B, S)
    with pytest.raises(tt.TTError) as e:
        tt.denoise_block_loop(B, S, V, tt.TT_F32, 0.1, 1.5, 3, S, tokens, masked, steps_used,
                              cstep, producer=producer, timeout_ms=50)
    assert e.value.status == tt.TT_ERR_TIMEOUT
    torch.cuda.synchronize()
    assert slept == [1]
    one = oracle.block_loop(B, S, fn, "f32", 0.1, 1.5, 3, S, stop_step=1)
    _compare(one, tokens, masked, steps_used, cstep)
    tt.denoise_block_loop(B, S, V, tt.TT_F32, 0.1, 1.5, 3, S, tokens, masked, steps_used, cstep,
                          producer=producer, start_step=1)
    torch.cuda.synchronize()
    _compare(oracle.block_loop(B, S, fn, "f32", 0.1, 1.5, 3, S), tokens, masked, steps_used, cstep)
