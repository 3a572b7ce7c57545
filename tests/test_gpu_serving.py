"""GPU parity of the many-stream configurations at their full model shapes:
several streams with ragged contexts decode frames together through the
layered step (tensor-core projections, grouped-query attention over the paged
cache, per-stream sampling).

Both configurations run at their full stream counts (16 and 128) with the
workloads' own seeded prompt lengths (32..256 and 256..2048), so the decode
takes the kernels the benchmark times (the serving step's 1,024 attention
CTAs pick the four-warp grouped-query kernel).

Checks, per configuration:
  * the streams with the shortest and the longest context against the oracle
    under teacher forcing (the serving configuration with the
    oracle's bf16 cache, as its cache is bf16): logits within 3e-2, argmax
    agreement >= 99.5%, and the drawn codes equal the float sampling rule
    applied to the GPU's own logits;
  * the shortest, the median and the longest stream decoded alone (one active
    stream, the same layered step),
    teacher-forced with the codes drawn inside the batch, give the same logits
    up to float reassociation -- a stream's result does not depend on the batch
    around it -- and each run's draws follow the float rule on its own logits.
    (The split-K projections add partial sums with float atomics, so logits
    vary in their last bits from run to run; a free-running sampled draw near a
    CDF boundary may then legitimately differ, which teacher forcing avoids.)
"""
import contextlib
import os

import numpy as np
import pytest

from autoregressive_tts_decode_gb300 import synth
from tests import parity_util as pu

pytestmark = pytest.mark.gpu

TOL_BF16 = 3e-2
FRAMES = 2

CASES = {
    # name: (workload, oracle cache in bf16)
    "serving128": ("serving128", True),
    "batched16": ("batched16", True),
}


@pytest.fixture(scope="module")
def q3():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from autoregressive_tts_decode_gb300 import build, q3tts
    build.build()
    return q3tts


@contextlib.contextmanager
def _layered_only():
    old = os.environ.get("Q3TTS_FRAME_KERNEL")
    os.environ["Q3TTS_FRAME_KERNEL"] = "0"
    try:
        yield
    finally:
        if old is None:
            del os.environ["Q3TTS_FRAME_KERNEL"]
        else:
            os.environ["Q3TTS_FRAME_KERNEL"] = old


@pytest.mark.parametrize("case", list(CASES))
def test_many_streams_full_shapes(q3, oracle_mod, case):
    import torch
    name, kv_bf16 = CASES[case]
    wl = synth.WORKLOADS[name]
    s = wl.shape
    lens = wl.prompt_lengths()
    assert len(lens) == wl.streams
    order = np.argsort(lens, kind="stable")
    checked = [int(order[0]), int(order[len(lens) // 2]), int(order[-1])]  # shortest, median, longest
    W, Wd = pu.gpu_weights(s, gen_device="cuda")
    prompts = synth.make_prompts(s, lens)
    ids = list(range(len(lens)))
    u = synth.uniforms(ids, FRAMES)
    eng = q3.Engine(s, Wd, max_streams=len(lens), kv_cap=wl.kv_cap, page_size=wl.page_size)
    codes, logits = pu.run_gpu(eng, ids, prompts, wl.sampling, FRAMES, uniforms=u)
    eng.close()
    # the shortest, the median and the longest stream alone, on the same layered step
    for k in checked:
        with _layered_only():
            one = q3.Engine(s, Wd, max_streams=1, kv_cap=wl.kv_cap, page_size=wl.page_size)
        c1, l1 = pu.run_gpu(one, [0], [prompts[k]], wl.sampling, FRAMES, uniforms=u[k:k + 1],
                            forced=codes[k:k + 1])
        one.close()
        # the same arithmetic up to fp32 reassociation (split-K atomics); with a
        # bf16 cache that can also send a cached k or v to the other bf16
        # neighbour (2^-8 relative), which moves logits by a few 1e-3
        same = 1e-2 if s.kv_dtype == synth.DTYPE_BF16 else 2e-3
        assert float(np.max(np.abs(l1[0] - logits[k]))) < same
        assert pu.sampler_replay(oracle_mod, s, wl.sampling, c1[0], l1[0], codes[k], u[k]) == 0
        assert pu.sampler_replay(oracle_mod, s, wl.sampling, codes[k], logits[k], codes[k], u[k]) == 0
    del Wd
    torch.cuda.empty_cache()
    # the shortest and the longest stream against the oracle (the oracle's
    # prefill of the longest prompt dominates this test's time)
    for k in (checked[0], checked[-1]):
        orc = oracle_mod.Oracle(s, W, 1, wl.kv_cap, kv_bf16=kv_bf16)
        oc, ol = pu.run_oracle(orc, 0, prompts[k].numpy(), wl.sampling, FRAMES, forced=codes[k], uniforms=u[k])
        del orc
        err, agree = pu.logits_report(logits[k], ol, s)
        assert err < TOL_BF16, (k, lens[k], err)
        assert agree >= 0.995, (k, lens[k], agree)
        assert pu.sampler_replay(oracle_mod, s, wl.sampling, codes[k], logits[k], codes[k], u[k]) == 0
