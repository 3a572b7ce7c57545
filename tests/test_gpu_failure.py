"""Failure detection on the GPU without a GPU fault.

Every device-side wait of the persistent frame kernel (ring slots, side slots,
the grid barrier) is bounded; when one runs out the kernel records
Q3TTS_ERR_TIMEOUT, raises its abort flag, lets its in-flight copies land and
returns, and q3tts_sync_status reports the code and clears the error and
barrier words.  The test hook q3tts_debug_fail_barrier makes one CTA leave out
its arrival at one grid barrier -- a flag that nothing else sets -- with the
frame's wait bound cut to 50 microseconds, so the other CTAs' waits run out.
No trap, assert, bad address or endless loop is involved.

After the failed frame the handle must be usable: another stream decodes on
exactly as the oracle does, and the failed stream decodes exactly once it is
prefilled again.
"""
import time

import numpy as np
import pytest

from autoregressive_tts_decode_gb300 import synth
from tests import parity_util as pu

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny"]


@pytest.fixture(scope="module")
def q3():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from autoregressive_tts_decode_gb300 import build, q3tts
    build.build()
    return q3tts


@pytest.fixture(scope="module")
def tiny_weights(q3):
    return pu.gpu_weights(TINY.shape)


def _one_frame(eng, sid, static):
    import torch
    u = torch.from_numpy(synth.uniforms([sid], 1)[:, 0]).cuda()
    c = torch.zeros((1, 16), dtype=torch.int32, device="cuda")
    if static:
        eng.step_frame_static(sid, TINY.sampling, u[0], c)
    else:
        eng.step_frame([sid], TINY.sampling, u, c)


def _exact_vs_oracle(eng, oracle_mod, W, sid, prompt, prefill):
    codes, logits = pu.run_gpu(eng, [sid], [prompt], TINY.sampling, 3,
                               uniforms=synth.uniforms([sid], 3), prefill=prefill)
    orc = oracle_mod.Oracle(TINY.shape, W, 2, 64)
    oc, ol = pu.run_oracle(orc, sid, prompt.numpy(), TINY.sampling, 3,
                           uniforms=synth.uniforms([sid], 3)[0])
    assert np.array_equal(codes[0], oc)
    assert np.max(np.abs(logits[0] - ol)) < 1e-4


@pytest.mark.parametrize("static", [False, True], ids=["step_frame", "step_frame_static"])
@pytest.mark.parametrize("barrier", [0, 9])
def test_skipped_arrival_times_out_and_handle_recovers(q3, oracle_mod, tiny_weights, static,
                                                       barrier):
    W, Wd = tiny_weights
    eng = q3.Engine(TINY.shape, Wd, max_streams=2, kv_cap=64)
    prompts = synth.make_prompts(TINY.shape, [16, 12])
    eng.prefill(0, prompts[0].cuda())
    eng.prefill(1, prompts[1].cuda())
    eng.sync()
    eng.debug_fail_barrier(barrier, 50)
    t0 = time.perf_counter()
    _one_frame(eng, 0, static)
    with pytest.raises(q3.Q3TTSError) as e:
        eng.sync()
    dt = time.perf_counter() - t0
    assert e.value.code == q3.ERR_TIMEOUT
    assert dt < 1.0, dt  # the 50 us bound, not the default of about 2 s, ended the waits
    eng.sync()  # the error word was cleared with the report
    # the other stream was not touched by the failed frame
    _exact_vs_oracle(eng, oracle_mod, W, 1, prompts[1], prefill=False)
    # the failed stream decodes exactly once restarted
    _exact_vs_oracle(eng, oracle_mod, W, 0, prompts[0], prefill=True)
    eng.close()


def test_arming_past_the_last_barrier_changes_nothing(q3, oracle_mod, tiny_weights):
    W, Wd = tiny_weights
    eng = q3.Engine(TINY.shape, Wd, max_streams=2, kv_cap=64)
    p = synth.make_prompts(TINY.shape, [16])[0]
    eng.prefill(0, p.cuda())
    eng.debug_fail_barrier(1 << 30, 200000)  # a bound no normal wait reaches
    _exact_vs_oracle(eng, oracle_mod, W, 0, p, prefill=False)
    with pytest.raises(q3.Q3TTSError) as e:
        eng.debug_fail_barrier(-1, 50)
    assert e.value.code == q3.ERR_ARG
    eng.close()
