"""The layered frame step replayed from a captured CUDA graph gives the same
frames as the same kernels launched one by one (Q3TTS_GRAPH=0): identical
codes, for free-running and teacher-forced steps, with changing input and
output buffers from call to call, a change of the active-stream count
(recapture), and the same number of kernels per step.  A step that asks for
a logits dump runs kernel by kernel; its codes agree with both."""
import contextlib
import os

import numpy as np
import pytest

from autoregressive_tts_decode_gb300 import synth
from tests import parity_util as pu

pytestmark = pytest.mark.gpu

FRAMES = 3


@pytest.fixture(scope="module")
def q3():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from autoregressive_tts_decode_gb300 import build, q3tts
    build.build()
    return q3tts


@contextlib.contextmanager
def _env(**kv):
    old = {k: os.environ.get(k) for k in kv}
    os.environ.update(kv)
    try:
        yield
    finally:
        for k, v in old.items():
            if v is None:
                del os.environ[k]
            else:
                os.environ[k] = v


def _run(q3, shape, W, prompts, schedule, graph, forced=None, dump=False):
    """Runs the (stream ids, frame) schedule; fresh device buffers every call."""
    import torch
    env = {"Q3TTS_FRAME_KERNEL": "0"} if graph else {"Q3TTS_FRAME_KERNEL": "0", "Q3TTS_GRAPH": "0"}
    with _env(**env):
        eng = q3.Engine(shape, W, max_streams=len(prompts), kv_cap=64)
    for sid, p in enumerate(prompts):
        eng.prefill(sid, p.to("cuda"))
    u_all = synth.uniforms(list(range(len(prompts))), len(schedule))
    width = shape.codec_vocab + 15 * shape.cp_vocab
    out = []
    l0 = eng.kernel_launches()
    per_step = []
    for k, ids in enumerate(schedule):
        u = torch.from_numpy(np.ascontiguousarray(u_all[ids, k])).to("cuda")
        c = torch.full((len(ids), 16), -1, dtype=torch.int32, device="cuda")
        fc = None if forced is None else torch.from_numpy(np.ascontiguousarray(forced[ids, k])).to("cuda")
        lg = torch.zeros((len(ids), width), dtype=torch.float32, device="cuda") if dump else None
        a = eng.kernel_launches()
        eng.step_frame(ids, synth.QWEN_DEFAULT_SAMPLING, u, c, forced=fc, logits=lg)
        per_step.append(eng.kernel_launches() - a)
        out.append(c.cpu().numpy())
    eng.sync()
    total = eng.kernel_launches() - l0
    eng.close()
    return out, per_step, total


def test_graph_replay_matches_kernel_by_kernel(q3):
    wl = synth.WORKLOADS["tiny"]
    shape = wl.shape
    _, W = pu.gpu_weights(shape)
    prompts = synth.make_prompts(shape, [16, 23, 9, 30])
    # 4 streams, then 2 (a new capture), then 4 again
    schedule = [[0, 1, 2, 3], [0, 1, 2, 3], [1, 3], [0, 1, 2, 3], [0, 1, 2, 3]]
    g, g_steps, g_total = _run(q3, shape, W, prompts, schedule, graph=True)
    k, k_steps, k_total = _run(q3, shape, W, prompts, schedule, graph=False)
    for a, b in zip(g, k):
        assert np.array_equal(a, b)
        assert (a >= 0).all()
    assert g_steps == k_steps and g_total == k_total
    d, _, _ = _run(q3, shape, W, prompts, schedule, graph=True, dump=True)
    for a, b in zip(d, k):
        assert np.array_equal(a, b)


def test_graph_replay_teacher_forced(q3):
    wl = synth.WORKLOADS["tiny"]
    shape = wl.shape
    _, W = pu.gpu_weights(shape)
    prompts = synth.make_prompts(shape, [12, 17, 20])
    rng = np.random.default_rng(3)
    forced = np.stack([rng.integers(0, shape.codec_vocab, size=(3, FRAMES)),
                       *[rng.integers(0, shape.cp_vocab, size=(3, FRAMES)) for _ in range(15)]], axis=-1)
    forced = forced.astype(np.int32)
    schedule = [[0, 1, 2]] * FRAMES
    g, _, _ = _run(q3, shape, W, prompts, schedule, graph=True, forced=forced)
    k, _, _ = _run(q3, shape, W, prompts, schedule, graph=False, forced=forced)
    for a, b in zip(g, k):
        assert np.array_equal(a, b)
