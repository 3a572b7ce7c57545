"""GPU parity of every branch of the sampling rule.

Controls of the "qwen3-tts-hip" README, section "Library Usage"
(GenerateOptions: do_sample, top_k, top_p, temperature, repetition_penalty and
their subtalker_* counterparts).  Each case decodes a few frames on the GPU,
then (1) replays every one of the frame's 16 draws through the oracle's float
rule on the logits the GPU drew from -- the picks must be identical -- and
(2) runs the oracle teacher-forced with the GPU's codes: logits within 1e-4
(fp32 weights and cache).

Branches covered: the top-p prefix (0.6 and 0.95); top-k 1, top-k off (0: the
whole vocabulary) and top-k 200 (wider than the persistent kernel's candidate
path, so the layered sampler's full sort); a repetition penalty of 1.3 over the
stream's history; a low temperature (0.05); and a head whose logits are all
equal, where every rank is a tie (lowest index first) and the persistent
kernel's candidate bound admits the whole vocabulary, so its bisection
fallback runs.  Each case runs on the persistent frame kernel where that path
takes the settings and on the layered step always.
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
RAGGED = dataclasses.replace(TINY.shape, talker_hidden=264, talker_ffn=776, cp_hidden=136,
                             cp_ffn=392, codec_vocab=3000, cp_vocab=1000)
TOL = 1e-4
FRAMES = 5

BASE = synth.QWEN_DEFAULT_SAMPLING


def _both(**kw):
    """The same controls for the semantic and the acoustic draws."""
    sub = {"sub_" + k: v for k, v in kw.items() if k in ("do_sample", "top_k", "top_p", "temperature")}
    return dataclasses.replace(BASE, **kw, **sub)


CASES = {
    "top_p_0.6": _both(top_p=0.6),
    "top_p_0.95": _both(top_p=0.95),
    "top_k_1": _both(top_k=1),
    "top_k_off": _both(top_k=0),
    "top_k_200": _both(top_k=200, top_p=0.9),
    "rep_1.3": dataclasses.replace(BASE, repetition_penalty=1.3),
    "rep_1.3_greedy": dataclasses.replace(synth.GREEDY, repetition_penalty=1.3),
    "T_0.05": _both(temperature=0.05),
}


@pytest.fixture(scope="module")
def q3():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from autoregressive_tts_decode_gb300 import build, q3tts
    build.build()
    return q3tts


@contextlib.contextmanager
def _frame_kernel(enabled: bool):
    old = os.environ.get("Q3TTS_FRAME_KERNEL")
    os.environ["Q3TTS_FRAME_KERNEL"] = "1" if enabled else "0"
    try:
        yield
    finally:
        if old is None:
            del os.environ["Q3TTS_FRAME_KERNEL"]
        else:
            os.environ["Q3TTS_FRAME_KERNEL"] = old


def _persistent_takes(sp):
    """Settings the persistent frame kernel draws itself (greedy or 1 <= top_k <= 64)."""
    def ok(do, k):
        return (not do) or 1 <= k <= 64
    return ok(sp.do_sample, sp.top_k) and ok(sp.sub_do_sample, sp.sub_top_k)


def _check(q3, oracle_mod, shape, W, Wd, sp, persistent):
    p = synth.make_prompts(shape, [19])[0]
    u = synth.uniforms([0], FRAMES)
    with _frame_kernel(persistent):
        eng = q3.Engine(shape, Wd, max_streams=1, kv_cap=40)
    eng.prefill(0, p.cuda())
    eng.sync()
    l0 = eng.kernel_launches()
    codes, logits = pu.run_gpu(eng, [0], [p], sp, FRAMES, uniforms=u, prefill=False)
    launches = eng.kernel_launches() - l0
    eng.close()
    if persistent and _persistent_takes(sp):
        assert launches == FRAMES, launches  # one persistent launch per frame
    else:
        assert launches > 50 * FRAMES, launches
    bad = pu.sampler_replay(oracle_mod, shape, sp, codes[0], logits[0], codes[0], u[0])
    assert bad == 0, bad
    orc = oracle_mod.Oracle(shape, W, 1, 40)
    _, ol = pu.run_oracle(orc, 0, p.numpy(), sp, FRAMES, forced=codes[0], uniforms=u[0])
    err, agree = pu.logits_report(logits[0], ol, shape)
    assert err < TOL, err
    return codes


@pytest.fixture(scope="module")
def weights(q3):
    return {"tiny": pu.gpu_weights(TINY.shape), "ragged": pu.gpu_weights(RAGGED)}


@pytest.mark.parametrize("persistent", [True, False], ids=["persistent", "layered"])
@pytest.mark.parametrize("shape_name", ["tiny", "ragged"])
@pytest.mark.parametrize("case", sorted(CASES))
def test_sampler_branch(q3, oracle_mod, weights, case, shape_name, persistent):
    shape = TINY.shape if shape_name == "tiny" else RAGGED
    W, Wd = weights[shape_name]
    _check(q3, oracle_mod, shape, W, Wd, CASES[case], persistent)


@pytest.mark.parametrize("persistent", [True, False], ids=["persistent", "layered"])
@pytest.mark.parametrize("sp_name", ["sampled", "greedy"])
def test_all_logits_tied(q3, oracle_mod, sp_name, persistent):
    """Zero codec and CodePredictor heads: every logit is 0.  Greedy draws take
    index 0; sampled draws keep ids 0..k-1 (lowest index first among equal
    values), weigh them equally and pick floor-like from the uniform -- all
    checked draw by draw against the oracle's float rule."""
    import torch
    shape = TINY.shape
    W = synth.make_weights(shape)
    W["talker.w_head"] = torch.zeros_like(W["talker.w_head"])
    W["cp.heads"] = torch.zeros_like(W["cp.heads"])
    Wd = {k: v.to("cuda") for k, v in W.items()}
    sp = BASE if sp_name == "sampled" else synth.GREEDY
    codes = _check(q3, oracle_mod, shape, W, Wd, sp, persistent)
    if sp_name == "greedy":
        assert not codes.any()
    else:
        assert codes.max() < sp.top_k and codes[0, :, 1:].max() < sp.sub_top_k
        assert len(np.unique(codes)) > 5  # the uniforms spread the picks
