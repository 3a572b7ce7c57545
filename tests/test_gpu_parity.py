"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle.

Frame structure per "Running Qwen3-TTS on an AMD R9700", section "Running
Qwen3-TTS"; sampling controls per the "qwen3-tts-hip" README, section "Library
Usage".  Tolerances: fp32 weights and cache (tiny shapes) 1e-4 on logits and
identical greedy codes; bf16 weights and cache (0.6B/1.7B shapes) 3e-2 on
logits with >= 99.5% argmax agreement under teacher forcing.  Sampled codes
must equal the oracle's float rule applied to the very logits the GPU drew
from (dumped through the logits output).
"""
import dataclasses

import numpy as np
import pytest

from autoregressive_tts_decode_gb300 import synth
from tests import parity_util as pu

pytestmark = pytest.mark.gpu

TINY = synth.WORKLOADS["tiny"]
TOL_F32 = 1e-4
TOL_BF16 = 3e-2


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


def _engine(q3, shape, Wd, streams=1, cap=64, **kw):
    return q3.Engine(shape, Wd, max_streams=streams, kv_cap=cap, **kw)


def test_tiny_prefill_pending_matches_oracle(q3, oracle_mod, tiny_weights):
    W, Wd = tiny_weights
    eng = _engine(q3, TINY.shape, Wd)
    p = synth.make_prompts(TINY.shape, [16])[0]
    eng.prefill(0, p.cuda())
    h, lg = eng.read_pending(0)
    orc = oracle_mod.Oracle(TINY.shape, W, 1, 64)
    orc.prefill(0, p.numpy())
    oh, ol = orc.pending(0)
    assert np.max(np.abs(h.cpu().numpy() - oh)) < TOL_F32
    assert np.max(np.abs(lg.cpu().numpy() - ol)) < TOL_F32
    assert eng.length(0) == 16


def test_tiny_greedy_codes_exact(q3, oracle_mod, tiny_weights):
    W, Wd = tiny_weights
    eng = _engine(q3, TINY.shape, Wd)
    p = synth.make_prompts(TINY.shape, [TINY.prompt_len])[0]
    codes, logits = pu.run_gpu(eng, [0], [p], TINY.sampling, TINY.frames)
    orc = oracle_mod.Oracle(TINY.shape, W, 1, 64)
    oc, ol = pu.run_oracle(orc, 0, p.numpy(), TINY.sampling, TINY.frames)
    assert np.array_equal(codes[0], oc)
    assert np.max(np.abs(logits[0] - ol)) < TOL_F32
    assert eng.length(0) == TINY.prompt_len + TINY.frames


def test_tiny_sampled_teacher_forced(q3, oracle_mod, tiny_weights):
    W, Wd = tiny_weights
    sp = synth.QWEN_DEFAULT_SAMPLING
    eng = _engine(q3, TINY.shape, Wd)
    p = synth.make_prompts(TINY.shape, [TINY.prompt_len])[0]
    u = synth.uniforms([0], 8)
    codes, logits = pu.run_gpu(eng, [0], [p], sp, 8, uniforms=u)
    orc = oracle_mod.Oracle(TINY.shape, W, 1, 64)
    oc, ol = pu.run_oracle(orc, 0, p.numpy(), sp, 8, forced=codes[0], uniforms=u[0])
    err, agree = pu.logits_report(logits[0], ol, TINY.shape)
    assert err < TOL_F32 and agree == 1.0
    assert pu.sampler_replay(oracle_mod, TINY.shape, sp, codes[0], logits[0], codes[0], u[0]) == 0


def test_teacher_forcing_feeds_forced_codes(q3, oracle_mod, tiny_weights):
    W, Wd = tiny_weights
    eng = _engine(q3, TINY.shape, Wd)
    p = synth.make_prompts(TINY.shape, [10])[0]
    rng = np.random.default_rng(3)
    forced = np.concatenate([rng.integers(0, TINY.shape.codec_vocab, (1, 4, 1)),
                             rng.integers(0, TINY.shape.cp_vocab, (1, 4, 15))], axis=2).astype(np.int32)
    codes, logits = pu.run_gpu(eng, [0], [p], TINY.sampling, 4, forced=forced)
    orc = oracle_mod.Oracle(TINY.shape, W, 1, 64)
    oc, ol = pu.run_oracle(orc, 0, p.numpy(), TINY.sampling, 4, forced=forced[0])
    assert np.max(np.abs(logits[0] - ol)) < TOL_F32
    assert np.array_equal(codes[0], oc)


RAGGED = dataclasses.replace(TINY.shape, talker_hidden=264, talker_ffn=776, cp_hidden=136,
                             cp_ffn=392, codec_vocab=3000, cp_vocab=1000)


def test_ragged_shapes_chunked_prefill(q3, oracle_mod):
    """Widths off the 256-element step, a projection (D_t != D_c), odd vocabularies,
    a prompt spanning two pages and three prefill chunks."""
    W, Wd = pu.gpu_weights(RAGGED)
    eng = q3.Engine(RAGGED, Wd, max_streams=1, kv_cap=40, prefill_chunk=10)
    p = synth.make_prompts(RAGGED, [23])[0]
    sp = synth.QWEN_DEFAULT_SAMPLING
    u = synth.uniforms([0], 6)
    codes, logits = pu.run_gpu(eng, [0], [p], sp, 6, uniforms=u)
    orc = oracle_mod.Oracle(RAGGED, W, 1, 40)
    oc, ol = pu.run_oracle(orc, 0, p.numpy(), sp, 6, forced=codes[0], uniforms=u[0])
    err, agree = pu.logits_report(logits[0], ol, RAGGED)
    assert err < TOL_F32 and agree == 1.0
    assert pu.sampler_replay(oracle_mod, RAGGED, sp, codes[0], logits[0], codes[0], u[0]) == 0


def test_batched_streams_match_single_stream_runs(q3, oracle_mod, tiny_weights):
    W, Wd = tiny_weights
    sp = synth.QWEN_DEFAULT_SAMPLING
    lens = [5, 17, 33]
    ids = [2, 0, 1]
    prompts = synth.make_prompts(TINY.shape, lens)
    u = synth.uniforms(ids, 5)
    eng = _engine(q3, TINY.shape, Wd, streams=3, cap=48)
    codes, logits = pu.run_gpu(eng, ids, prompts, sp, 5, uniforms=u)
    for b, sid in enumerate(ids):
        single = _engine(q3, TINY.shape, Wd, streams=3, cap=48)
        c1, l1 = pu.run_gpu(single, [sid], [prompts[b]], sp, 5, uniforms=u[b:b + 1])
        assert np.array_equal(c1[0], codes[b])
        assert np.max(np.abs(l1[0] - logits[b])) < 1e-5
        orc = oracle_mod.Oracle(TINY.shape, W, 3, 48)
        oc, ol = pu.run_oracle(orc, sid, prompts[b].numpy(), sp, 5, forced=codes[b], uniforms=u[b])
        err, agree = pu.logits_report(logits[b], ol, TINY.shape)
        assert err < TOL_F32 and agree == 1.0
        assert pu.sampler_replay(oracle_mod, TINY.shape, sp, codes[b], logits[b], codes[b], u[b]) == 0


def test_paged_pool_shared_and_reset(q3, tiny_weights):
    """A pool smaller than max_streams full streams: pages come back on reset."""
    W, Wd = tiny_weights
    eng = q3.Engine(TINY.shape, Wd, max_streams=2, kv_cap=64, kv_pages=5)
    p = synth.make_prompts(TINY.shape, [40, 40])
    eng.prefill(0, p[0].cuda())  # 3 pages
    with pytest.raises(q3.Q3TTSError) as e:
        eng.prefill(1, p[1].cuda())  # needs 3, 2 left
    assert e.value.code == q3.ERR_CAPACITY
    eng.reset(0)
    eng.prefill(1, p[1].cuda())
    eng.sync()


def _full_size(q3, oracle_mod, wl, frames):
    import torch
    s = wl.shape
    W, Wd = pu.gpu_weights(s, gen_device="cuda")
    p = synth.make_prompts(s, [wl.prompt_len])[0]
    u = synth.uniforms([0], frames)
    eng = q3.Engine(s, Wd, max_streams=1, kv_cap=wl.kv_cap)
    codes, logits = pu.run_gpu(eng, [0], [p], wl.sampling, frames, uniforms=u)
    eng.close()
    del Wd
    torch.cuda.empty_cache()
    orc = oracle_mod.Oracle(s, W, 1, wl.kv_cap)
    oc, ol = pu.run_oracle(orc, 0, p.numpy(), wl.sampling, frames, forced=codes[0], uniforms=u[0])
    err, agree = pu.logits_report(logits[0], ol, s)
    return codes, logits, oc, ol, err, agree, u


def test_06b_full_size_teacher_forced(q3, oracle_mod):
    wl = synth.WORKLOADS["0.6b"]
    codes, logits, oc, ol, err, agree, u = _full_size(q3, oracle_mod, wl, 3)
    assert err < TOL_BF16, err
    assert agree >= 0.995, agree
    assert pu.sampler_replay(oracle_mod, wl.shape, wl.sampling, codes[0], logits[0], codes[0], u[0]) == 0


def test_17b_full_size_teacher_forced(q3, oracle_mod):
    wl = synth.WORKLOADS["1.7b"]
    codes, logits, oc, ol, err, agree, u = _full_size(q3, oracle_mod, wl, 2)
    assert err < TOL_BF16, err
    assert agree >= 0.995, agree
    assert pu.sampler_replay(oracle_mod, wl.shape, wl.sampling, codes[0], logits[0], codes[0], u[0]) == 0


def test_errors_are_status_codes(q3, tiny_weights):
    import torch
    W, Wd = tiny_weights
    eng = _engine(q3, TINY.shape, Wd, streams=2, cap=20)
    u = torch.zeros((1, 16), dtype=torch.float32, device="cuda")
    c = torch.zeros((1, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(q3.Q3TTSError) as e:
        eng.step_frame([0], TINY.sampling, u, c)
    assert e.value.code == q3.ERR_STATE
    with pytest.raises(q3.Q3TTSError) as e:
        eng.prefill(0, torch.zeros((20, TINY.shape.talker_hidden), device="cuda"))
    assert e.value.code == q3.ERR_CAPACITY
    with pytest.raises(q3.Q3TTSError) as e:
        eng.prefill(5, torch.zeros((3, TINY.shape.talker_hidden), device="cuda"))
    assert e.value.code == q3.ERR_ARG
    eng.prefill(0, synth.make_prompts(TINY.shape, [18])[0].cuda())
    eng.step_frame([0], TINY.sampling, u, c)
    eng.step_frame([0], TINY.sampling, u, c)
    with pytest.raises(q3.Q3TTSError) as e:
        eng.step_frame([0], TINY.sampling, u, c)
    assert e.value.code == q3.ERR_CAPACITY
    bad = dataclasses.replace(synth.QWEN_DEFAULT_SAMPLING, temperature=0.0)
    eng.prefill(1, synth.make_prompts(TINY.shape, [4])[0].cuda())
    with pytest.raises(q3.Q3TTSError) as e:
        eng.step_frame([1], bad, u, c)
    assert e.value.code == q3.ERR_ARG
    u2 = torch.zeros((2, 16), dtype=torch.float32, device="cuda")
    c2 = torch.zeros((2, 16), dtype=torch.int32, device="cuda")
    with pytest.raises(q3.Q3TTSError) as e:
        eng.step_frame([1, 1], TINY.sampling, u2, c2)
    assert e.value.code == q3.ERR_ARG
    # an out-of-range forced code is reported by the device, memory stays safe
    f = torch.full((1, 16), 99999, dtype=torch.int32, device="cuda")
    eng.step_frame([1], TINY.sampling, u, c, forced=f)
    with pytest.raises(q3.Q3TTSError) as e:
        eng.sync()
    assert e.value.code == q3.ERR_ARG
    eng.sync()


def _with_frame_kernel(enabled: bool):
    import contextlib
    import os

    @contextlib.contextmanager
    def cm():
        old = os.environ.get("Q3TTS_FRAME_KERNEL")
        os.environ["Q3TTS_FRAME_KERNEL"] = "1" if enabled else "0"
        try:
            yield
        finally:
            if old is None:
                del os.environ["Q3TTS_FRAME_KERNEL"]
            else:
                os.environ["Q3TTS_FRAME_KERNEL"] = old
    return cm()


@pytest.mark.parametrize("shape_name", ["tiny", "ragged"])
def test_persistent_kernel_matches_layered_step(q3, oracle_mod, shape_name):
    """Batch-1 frames run as one persistent launch; the one-kernel-per-operation
    step, teacher-forced with the persistent kernel's codes, produces the same
    logits (fp32 reassociation only), and each path's draws follow the float
    rule on its own logits."""
    shape = TINY.shape if shape_name == "tiny" else RAGGED
    W, Wd = pu.gpu_weights(shape)
    sp = synth.QWEN_DEFAULT_SAMPLING
    p = synth.make_prompts(shape, [21])[0]
    u = synth.uniforms([0], 6)
    out = {}
    forced = None
    for fk in (True, False):
        with _with_frame_kernel(fk):
            eng = q3.Engine(shape, Wd, max_streams=1, kv_cap=40)
        eng.prefill(0, p.cuda())
        eng.sync()
        l0 = eng.kernel_launches()
        codes, logits = pu.run_gpu(eng, [0], [p], sp, 6, uniforms=u, prefill=False, forced=forced)
        out[fk] = (codes, logits, eng.kernel_launches() - l0)
        eng.close()
        forced = codes
    assert out[True][2] == 6, out[True][2]        # one launch per frame
    assert out[False][2] > 100 * 6
    assert np.max(np.abs(out[True][1] - out[False][1])) < 2e-5
    for fk in (True, False):
        codes, logits, _ = out[fk]
        assert pu.sampler_replay(oracle_mod, shape, sp, codes[0], logits[0], out[True][0][0], u[0]) == 0


def test_page_size_off_powers_of_two_takes_the_layered_step(q3, oracle_mod, tiny_weights):
    """The persistent kernel splits cache positions by shift and mask, so it is
    set up for power-of-two page sizes only; a 12-position page decodes through
    the one-kernel-per-operation step, with the same greedy codes as the oracle
    (the prompt spans two pages, the frames a third)."""
    W, Wd = tiny_weights
    p = synth.make_prompts(TINY.shape, [21])[0]
    frames = 6
    orc = oracle_mod.Oracle(TINY.shape, W, 1, 64)
    oc, ol = pu.run_oracle(orc, 0, p.numpy(), synth.GREEDY, frames)
    per_frame = {}
    for ps in (16, 12):
        eng = _engine(q3, TINY.shape, Wd, cap=64, page_size=ps)
        eng.prefill(0, p.cuda())
        eng.sync()
        l0 = eng.kernel_launches()
        codes, logits = pu.run_gpu(eng, [0], [p], synth.GREEDY, frames, prefill=False)
        per_frame[ps] = (eng.kernel_launches() - l0) / frames
        eng.close()
        assert np.array_equal(codes[0], oc), ps
        assert np.max(np.abs(logits[0] - ol)) < TOL_F32, ps
    assert per_frame[16] == 1          # one persistent launch per frame
    assert per_frame[12] > 1           # the layered step


@pytest.mark.parametrize("kv", ["f32", "bf16"])
def test_long_contexts_split_attention(q3, oracle_mod, tiny_weights, kv):
    """Streams whose contexts span several 64-position spans: the layered step and a
    chunked prefill take the split-context attention (tiny shapes: head_dim 64, two
    q heads per kv head), with an fp32 cache and with a bf16 cache (the oracle then
    rounds k and v to bf16 as they enter its cache)."""
    W, Wd = tiny_weights
    shape = TINY.shape if kv == "f32" else dataclasses.replace(TINY.shape, kv_dtype=synth.DTYPE_BF16)
    tol = TOL_F32 if kv == "f32" else 1e-3
    sp = synth.QWEN_DEFAULT_SAMPLING
    lens = [70, 300, 129]  # 2, 5 and 3 spans; the prefill runs in chunks of 128
    ids = [0, 1, 2]
    prompts = synth.make_prompts(shape, lens)
    u = synth.uniforms(ids, 4)
    eng = q3.Engine(shape, Wd, max_streams=3, kv_cap=512, prefill_chunk=128)
    codes, logits = pu.run_gpu(eng, ids, prompts, sp, 4, uniforms=u)
    eng.close()
    for b, sid in enumerate(ids):
        orc = oracle_mod.Oracle(shape, W, 1, 512, kv_bf16=(kv == "bf16"))
        oc, ol = pu.run_oracle(orc, 0, prompts[b].numpy(), sp, 4, forced=codes[b], uniforms=u[b])
        err, agree = pu.logits_report(logits[b], ol, shape)
        assert err < tol and agree == 1.0, (lens[b], err, agree)
        assert pu.sampler_replay(oracle_mod, shape, sp, codes[b], logits[b], codes[b], u[b]) == 0


def test_prefill_tensor_core_attention_17b_bf16_cache(q3, oracle_mod):
    """Chunked prefill at the 1.7B shapes with a bf16 cache: the causal attention
    of each chunk runs as 64-token query tiles on the tensor cores.  A 300-position
    prompt in chunks of 128 (later chunks start past position 0, the last query
    tile is ragged) against the oracle with the bf16 cache: pending hidden and
    logits after the prompt, and two teacher-forced frames."""
    import torch
    wl = synth.WORKLOADS["1.7b"]
    s = synth.SHAPE_17B_KV16
    W, Wd = pu.gpu_weights(s, gen_device="cuda")
    p = synth.make_prompts(s, [300])[0]
    eng = q3.Engine(s, Wd, max_streams=1, kv_cap=512, prefill_chunk=128)
    eng.prefill(0, p.cuda())
    hp, lp = eng.read_pending(0)
    hp, lp = hp.cpu().numpy(), lp.cpu().numpy()
    u = synth.uniforms([0], 2)
    codes, logits = pu.run_gpu(eng, [0], [p], wl.sampling, 2, uniforms=u)
    eng.close()
    del Wd
    torch.cuda.empty_cache()
    orc = oracle_mod.Oracle(s, W, 1, 512, kv_bf16=True)
    orc.prefill(0, p.numpy())
    oh, ol0 = orc.pending(0)
    assert np.max(np.abs(lp - ol0)) < TOL_BF16, np.max(np.abs(lp - ol0))
    assert np.max(np.abs(hp - oh)) < 0.05, np.max(np.abs(hp - oh))
    oc, ol = pu.run_oracle(orc, 0, p.numpy(), wl.sampling, 2, forced=codes[0], uniforms=u[0])
    err, agree = pu.logits_report(logits[0], ol, s)
    assert err < TOL_BF16, err
    assert agree >= 0.995, agree
