"""q3tts_step_frame_static: the batch-1 frame with its scratch in the library's
static device array gives the same frame as q3tts_step_frame (whose scratch is
in the handle's workspace), on two frames in a row, through the C ABI.

The file name keeps it last in collection so that it also runs after every
other GPU test in the same process (the static array is per process and is
shared by every handle); it must pass as well when run alone in a fresh
process."""
import dataclasses

import numpy as np
import pytest

from autoregressive_tts_decode_gb300 import synth
from tests import parity_util as pu

pytestmark = pytest.mark.gpu

FRAMES = 2


@pytest.fixture(scope="module")
def q3():
    import torch
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from autoregressive_tts_decode_gb300 import build, q3tts
    build.build()
    return q3tts


def _frames(eng, step, sp, u, forced=None):
    """Runs FRAMES frames of stream 0 through `step`; returns codes, logits."""
    import torch
    s = eng.shape
    width = s.codec_vocab + 15 * s.cp_vocab
    c = torch.zeros((1, 16), dtype=torch.int32, device="cuda")
    lg = torch.zeros((1, width), dtype=torch.float32, device="cuda")
    codes = np.zeros((FRAMES, 16), dtype=np.int32)
    logits = np.zeros((FRAMES, width), dtype=np.float32)
    for f in range(FRAMES):
        uf = torch.from_numpy(np.ascontiguousarray(u[:, f])).cuda()
        fc = None if forced is None else torch.from_numpy(np.ascontiguousarray(forced[f:f + 1])).cuda()
        step(eng, sp, uf, c, fc, lg)
        codes[f] = c.cpu().numpy()[0]
        logits[f] = lg.cpu().numpy()[0]
    eng.sync()
    return codes, logits


def _existing(eng, sp, u, c, fc, lg):
    eng.step_frame([0], sp, u, c, forced=fc, logits=lg)


def _static(eng, sp, u, c, fc, lg):
    eng.step_frame_static(0, sp, u[0], c, forced=fc, logits=lg)


@pytest.mark.parametrize("name,tol", [("tiny", 2e-5), ("0.6b", 1e-2)])
def test_static_scratch_frame_matches_step_frame(q3, oracle_mod, name, tol):
    """Stream A runs two frames through q3tts_step_frame; stream B, on another
    handle with the same weights and prompt, runs them through
    q3tts_step_frame_static, teacher-forced with A's codes.  Both run the same
    kernel, so the logits agree up to float-atomic reassociation (tiny fp32:
    2e-5; 0.6B, bf16 weights and Talker cache: 1e-2, as reassociation can also
    send a cached k or v to the other bf16 neighbour -- measured 0.0026 -- well
    inside the 3e-2 parity bound), and B's draws follow the float sampling rule
    on B's own logits.  With an fp32 cache the codes agree too; with a bf16 one
    a draw whose uniform sits near a boundary of the cumulative weights may go
    the other way (B is teacher-forced, so its state does not follow its draws)."""
    wl = synth.WORKLOADS[name]
    shape = wl.shape
    W, Wd = pu.gpu_weights(shape, gen_device="cuda" if name != "tiny" else "cpu")
    sp = synth.QWEN_DEFAULT_SAMPLING
    p = synth.make_prompts(shape, [wl.prompt_len or 16])[0].cuda()
    u = synth.uniforms([0], FRAMES)
    out = {}
    for key, step in (("existing", _existing), ("static", _static)):
        eng = q3.Engine(shape, Wd, max_streams=1, kv_cap=128)
        eng.prefill(0, p)
        eng.sync()
        l0 = eng.kernel_launches()
        forced = None if key == "existing" else out["existing"][0]
        codes, logits = _frames(eng, step, sp, u, forced)
        out[key] = (codes, logits, eng.kernel_launches() - l0, eng.length(0))
        eng.close()
    (ca, la, na, lena), (cb, lb, nb, lenb) = out["existing"], out["static"]
    assert na == FRAMES and nb == FRAMES          # one persistent launch per frame
    assert lena == lenb == p.shape[0] + FRAMES
    err = float(np.max(np.abs(la - lb)))
    assert err < tol, err
    if shape.kv_dtype == synth.DTYPE_F32:
        assert np.array_equal(ca, cb)
    assert pu.sampler_replay(oracle_mod, shape, sp, cb, lb, ca, u[0]) == 0


def test_static_scratch_rejections_leave_state(q3):
    """Requests the static path cannot take return their error before any launch
    and leave the stream where it was; the stream then decodes normally."""
    import torch
    wl = synth.WORKLOADS["tiny"]
    shape = wl.shape
    _, Wd = pu.gpu_weights(shape)
    eng = q3.Engine(shape, Wd, max_streams=1, kv_cap=64)
    p = synth.make_prompts(shape, [16])[0].cuda()
    u = torch.zeros(16, dtype=torch.float32, device="cuda")
    c = torch.zeros(16, dtype=torch.int32, device="cuda")
    sp = synth.QWEN_DEFAULT_SAMPLING
    with pytest.raises(q3.Q3TTSError) as e:
        eng.step_frame_static(0, sp, u, c)
    assert e.value.code == q3.ERR_STATE
    eng.prefill(0, p)
    wide_k = dataclasses.replace(sp, top_k=200)    # beyond the kernel's candidate path
    with pytest.raises(q3.Q3TTSError) as e:
        eng.step_frame_static(0, wide_k, u, c)
    assert e.value.code == q3.ERR_UNSUPPORTED
    with pytest.raises(q3.Q3TTSError) as e:
        eng.step_frame_static(1, sp, u, c)             # no such stream
    assert e.value.code == q3.ERR_ARG
    assert eng.length(0) == 16
    l0 = eng.kernel_launches()
    eng.step_frame_static(0, sp, u, c)
    eng.sync()
    assert eng.length(0) == 17 and eng.kernel_launches() == l0 + 1
    eng.close()


def test_static_scratch_too_small_is_rejected(q3):
    """A shape the persistent kernel accepts whose scratch exceeds the static
    array: 128 query heads over 64 KV heads of width 128 (wide QKV rows and
    many attention partials) with a 4096-entry CodePredictor vocabulary.  The
    call returns Q3TTS_ERR_SCRATCH before anything is launched (configuration
    checks come before the stream's state)."""
    import torch
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    shape = dataclasses.replace(synth.WORKLOADS["tiny"].shape, talker_layers=1, cp_layers=1,
                                talker_hidden=2048, cp_hidden=1024, talker_ffn=256, cp_ffn=256,
                                n_q_heads=128, n_kv_heads=64, head_dim=128, codec_vocab=256,
                                cp_vocab=4096, weight_dtype=synth.DTYPE_BF16)
    ncta = min(n_sm, 256)
    cpg = max(1, ncta // 64)

    def al(x):
        return (x + 255) // 256 * 256
    xst = max(2048, 2 * 1024)
    qkv_rows = (128 + 2 * 64) * 128
    # barrier words, residual base / attention / FFN buffers, then the tagged
    # words (8 bytes each): QKV rows, projection, attention partials, logits
    need = 256 + al(4 * 2 * xst) * 2 + al(4 * 2 * 4 * xst) + al(8 * 2 * qkv_rows) + al(8 * 2 * 1024) \
        + al(8 * 128 * cpg * 130) + al(8 * 4096)
    if need <= q3.STATIC_SCRATCH_BYTES:
        pytest.skip(f"{n_sm} SMs: this shape's scratch fits the static array")
    _, Wd = pu.gpu_weights(shape, gen_device="cuda")
    eng = q3.Engine(shape, Wd, max_streams=1, kv_cap=32)
    u = torch.zeros(16, dtype=torch.float32, device="cuda")
    c = torch.zeros(16, dtype=torch.int32, device="cuda")
    l0 = eng.kernel_launches()
    with pytest.raises(q3.Q3TTSError) as e:
        eng.step_frame_static(0, synth.QWEN_DEFAULT_SAMPLING, u, c)
    assert e.value.code == q3.ERR_SCRATCH
    assert "static scratch" in str(e.value)
    assert eng.kernel_launches() == l0 and eng.length(0) == 0
    eng.close()
