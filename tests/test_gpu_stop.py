"""GPU parity of the stop conditions: the end-of-stream code and the masking of
special semantic codes, on the persistent kernel (q3tts_step_frame and the
static-scratch step) and on the layered step, against the oracle.

The pages leave end-of-stream handling open ("qwen3-tts-hip" README, "Status":
EOS behaviour still needs parity work); the reading adopted: semantic codes >=
special_from other than eos_token are never drawn; a frame whose fed semantic
code is eos_token yields [c0, -1 x 15] and ends the stream; later frames yield
sixteen -1; a prefill restarts the stream.
"""
import contextlib
import dataclasses
import os

import numpy as np
import pytest

from autoregressive_tts_decode_gb300 import synth
from tests import parity_util as pu

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny"]
SPECIAL = 2048  # codec codes 2048..3071 are special
EOS = 2150
SP = dataclasses.replace(synth.QWEN_DEFAULT_SAMPLING, eos_token=EOS, special_from=SPECIAL)
FRAMES = 5
EOS_FRAME = 2


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


@contextlib.contextmanager
def _env(name, value):
    old = os.environ.get(name)
    os.environ[name] = value
    try:
        yield
    finally:
        if old is None:
            del os.environ[name]
        else:
            os.environ[name] = old


def _engine(q3, Wd, path):
    if path == "layered":
        with _env("Q3TTS_FRAME_KERNEL", "0"):
            return q3.Engine(TINY.shape, Wd, max_streams=2, kv_cap=64)
    return q3.Engine(TINY.shape, Wd, max_streams=2, kv_cap=64)


def _run(eng, path, prompt, forced, u):
    """Frames of stream 0 one at a time (static path: q3tts_step_frame_static)."""
    import torch
    if path != "static":
        return pu.run_gpu(eng, [0], [prompt], SP, FRAMES, forced=forced[None], uniforms=u[None])
    s = TINY.shape
    eng.prefill(0, prompt.cuda())
    width = s.codec_vocab + 15 * s.cp_vocab
    codes = np.zeros((1, FRAMES, 16), dtype=np.int32)
    logits = np.zeros((1, FRAMES, width), dtype=np.float32)
    c = torch.zeros((1, 16), dtype=torch.int32, device="cuda")
    lg = torch.zeros((1, width), dtype=torch.float32, device="cuda")
    for f in range(FRAMES):
        uu = torch.from_numpy(np.ascontiguousarray(u[f])).cuda()
        fc = torch.from_numpy(np.ascontiguousarray(forced[f])).cuda()
        eng.step_frame_static(0, SP, uu, c, forced=fc, logits=lg)
        codes[0, f] = c.cpu().numpy()
        logits[0, f] = lg.cpu().numpy()
    eng.sync()
    return codes, logits


@pytest.mark.parametrize("path", ["persistent", "static", "layered"])
def test_end_of_stream_and_masking(q3, oracle_mod, tiny_weights, path):
    W, Wd = tiny_weights
    prompt = synth.make_prompts(TINY.shape, [16])[0]
    u = synth.uniforms([0], FRAMES)[0]
    # the trajectory: the oracle's own draws (with masking), the end-of-stream
    # code fed at frame EOS_FRAME
    orc = oracle_mod.Oracle(TINY.shape, W, 1, 64)
    free, _ = pu.run_oracle(orc, 0, prompt.numpy(), SP, FRAMES, uniforms=u)
    assert (free[:, 0] < SPECIAL).all() or (free[:, 0] == EOS).any()
    forced = free.copy()
    forced[EOS_FRAME, 0] = EOS
    forced[EOS_FRAME + 1:] = 0  # ignored once the stream has ended
    oc, ol = pu.run_oracle(orc, 0, prompt.numpy(), SP, FRAMES, forced=forced, uniforms=u)
    assert (oc[EOS_FRAME, 1:] == -1).all() and (oc[EOS_FRAME + 1:] == -1).all()

    eng = _engine(q3, Wd, path)
    codes, logits = _run(eng, path, prompt, forced, u)
    g = codes[0]
    # frames up to the end: logits as the oracle's, draws by the masked float rule
    n = EOS_FRAME + 1
    assert np.max(np.abs(logits[0, :n, :TINY.shape.codec_vocab] - ol[:n, :TINY.shape.codec_vocab])) < 1e-4
    assert np.max(np.abs(logits[0, :EOS_FRAME] - ol[:EOS_FRAME])) < 1e-4
    assert pu.sampler_replay(oracle_mod, TINY.shape, SP, g[:EOS_FRAME], logits[0, :EOS_FRAME],
                             forced[:EOS_FRAME], u[:EOS_FRAME]) == 0
    # the end-of-stream frame keeps its drawn semantic code (masked rule), then -1
    c_eos = oracle_mod.sample(logits[0, EOS_FRAME, :TINY.shape.codec_vocab], True, SP.top_k, SP.top_p,
                              SP.temperature, SP.repetition_penalty,
                              np.isin(np.arange(TINY.shape.codec_vocab), forced[:EOS_FRAME, 0]).astype(np.uint8),
                              float(u[EOS_FRAME, 0]), special_from=SPECIAL, eos_token=EOS)
    assert g[EOS_FRAME, 0] == c_eos
    assert (g[EOS_FRAME, 1:] == -1).all()
    assert (g[EOS_FRAME + 1:] == -1).all()
    assert (g[:EOS_FRAME, 0] < SPECIAL).all()
    assert eng.finished(0) and not eng.finished(1)
    # a prefill restarts the stream: its frames draw codes again, by the same rule
    codes2, logits2 = _run(eng, path, prompt, forced, u)
    assert (codes2[0, :EOS_FRAME] >= 0).all() and (codes2[0, EOS_FRAME + 1:] == -1).all()
    assert pu.sampler_replay(oracle_mod, TINY.shape, SP, codes2[0, :EOS_FRAME], logits2[0, :EOS_FRAME],
                             forced[:EOS_FRAME], u[:EOS_FRAME]) == 0
    eng.reset(0)
    assert not eng.finished(0)
    eng.close()


def test_masked_greedy_and_disabled_top_k_layered(q3, oracle_mod, tiny_weights):
    """Greedy and top-k disabled (k = 0: all allowed codes kept) with masking, on
    the layered step (two streams): every semantic draw follows the masked rule."""
    W, Wd = tiny_weights
    prompts = synth.make_prompts(TINY.shape, [12, 9])
    for sp in (dataclasses.replace(SP, do_sample=False, eos_token=-1),
               dataclasses.replace(SP, top_k=0, eos_token=-1)):
        u = synth.uniforms([0, 1], 4)
        eng = q3.Engine(TINY.shape, Wd, max_streams=2, kv_cap=64)
        codes, logits = pu.run_gpu(eng, [0, 1], prompts, sp, 4, uniforms=u)
        eng.close()
        for b in range(2):
            assert (codes[b, :, 0] < SPECIAL).all()
            assert pu.sampler_replay(oracle_mod, TINY.shape, sp, codes[b], logits[b], codes[b], u[b]) == 0
