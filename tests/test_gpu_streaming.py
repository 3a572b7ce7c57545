"""GPU tests of frame-incremental streaming (q3tts_step_frames and
q3tts_frames_ready; the counterpart of the engine's streaming session,
"qwen3-tts-hip" README, "Library Usage": start_stream, then next_audio_chunk).

A chunk runs each frame exactly as q3tts_step_frame would, so chunked decoding
yields the same codes as frame-by-frame decoding (greedy, tiny fp32 shapes:
deterministic) and as the oracle; the codes reach the pinned host buffer frame
by frame; a frame that cannot be enqueued stops the chunk with its error code.
"""
import numpy as np
import pytest

from autoregressive_tts_decode_gb300 import synth
from tests import parity_util as pu

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny"]
SP = synth.GREEDY


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


def _uniforms(ids, frames):
    import torch
    u = synth.uniforms(ids, frames)  # [n, frames, 16]
    return torch.from_numpy(np.ascontiguousarray(u.transpose(1, 0, 2))).cuda()  # [frames, n, 16]


@pytest.mark.parametrize("ids,chunk", [([0], 4), ([0, 1], 3)], ids=["persistent", "layered"])
def test_chunks_equal_frame_by_frame_and_oracle(q3, oracle_mod, tiny_weights, ids, chunk):
    W, Wd = tiny_weights
    frames = 10
    prompts = synth.make_prompts(TINY.shape, [16, 11][:len(ids)])
    eng = q3.Engine(TINY.shape, Wd, max_streams=2, kv_cap=64)
    ref, _ = pu.run_gpu(eng, ids, prompts, SP, frames)  # frame by frame
    for sid, p in zip(ids, prompts):
        eng.prefill(sid, p.cuda())
    got = np.concatenate(list(eng.stream_codes(ids, SP, _uniforms(ids, frames), chunk)), axis=0)
    eng.close()
    assert got.shape == (frames, len(ids), 16)
    for b, sid in enumerate(ids):
        assert np.array_equal(got[:, b], ref[b])
        orc = oracle_mod.Oracle(TINY.shape, W, 2, 64)
        oc, _ = pu.run_oracle(orc, sid, prompts[b].numpy(), SP, frames)
        assert np.array_equal(got[:, b], oc)


def test_frames_ready_and_host_copies(q3, tiny_weights):
    import torch
    _, Wd = tiny_weights
    eng = q3.Engine(TINY.shape, Wd, max_streams=1, kv_cap=64)
    eng.prefill(0, synth.make_prompts(TINY.shape, [16])[0].cuda())
    F = 6
    codes = torch.full((F, 1, 16), -7, dtype=torch.int32, device="cuda")
    host = torch.full((F, 1, 16), -7, dtype=torch.int32).pin_memory()
    eng.step_frames([0], SP, _uniforms([0], F), codes, codes_host=host)
    assert 0 <= eng.frames_ready() <= F
    eng.sync()
    assert eng.frames_ready() == F
    assert np.array_equal(host.numpy(), codes.cpu().numpy())
    assert (host.numpy() >= 0).all()
    assert eng.length(0) == 16 + F
    eng.close()


def test_chunk_stops_at_capacity(q3, tiny_weights):
    """A cache of 24 positions after a 20-position prompt holds four more frames:
    the fifth frame of an eight-frame chunk is refused before launch, and the
    chunk counts the four enqueued ones."""
    import torch
    _, Wd = tiny_weights
    eng = q3.Engine(TINY.shape, Wd, max_streams=1, kv_cap=24)
    eng.prefill(0, synth.make_prompts(TINY.shape, [20])[0].cuda())
    F = 8
    codes = torch.zeros((F, 1, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(q3.Q3TTSError) as e:
        eng.step_frames([0], SP, _uniforms([0], F), codes)
    assert e.value.code == q3.ERR_CAPACITY
    eng.sync()
    assert eng.frames_ready() == 4
    assert eng.length(0) == 24
    with pytest.raises(q3.Q3TTSError) as e:
        eng.step_frames([0], SP, _uniforms([0], q3.MAX_CHUNK + 1), torch.zeros((q3.MAX_CHUNK + 1, 1, 16),
                                                                                dtype=torch.int32, device="cuda"))
    assert e.value.code == q3.ERR_ARG
    eng.close()
