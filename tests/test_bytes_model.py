"""Pins of the byte model against the numbers printed in "Running Qwen3-TTS on
an AMD R9700" (flynnbody.com), section "Running Qwen3-TTS": module sizes
(CodePredictor 0.350 GB in fp16), the per-frame closed form 3.483 + 15 x 0.350 =
8.733 GB, 640 GB/s / 8.733 GB = 73.3 frames/s, RTF ~0.17 and ~5.9x real time;
and the frame constants (24 kHz / 1,920 samples = 12.5 frames/s)."""
import json
import os

import pytest

from autoregressive_tts_decode_gb300 import bytes_model as bm
from autoregressive_tts_decode_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "r9700_frame_cost.json")


def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_frame_constants():
    g = golden()
    assert synth.SAMPLE_RATE / synth.SAMPLES_PER_FRAME == g["frames_per_second_realtime"]
    assert synth.N_CODEBOOKS == g["codebook_tokens_per_frame"]
    assert synth.SAMPLES_PER_FRAME / synth.SAMPLE_RATE == pytest.approx(g["frame_seconds"])


def test_codepredictor_module_size_matches_page():
    g = golden()
    cp = bm.module_bytes(synth.SHAPE_17B)["code_predictor"]
    assert cp / 1e9 == pytest.approx(g["codepredictor_gb_fp16"], abs=0.0006)


def test_page_closed_form_arithmetic():
    g = golden()
    per_frame = bm.page_frame_bytes(g["talker_gb_fp16"], g["codepredictor_gb_fp16"])
    assert per_frame == pytest.approx(g["bytes_per_frame_gb"], abs=5e-4)
    fps = g["r9700_bandwidth_gbs"] / per_frame
    assert fps == pytest.approx(g["bandwidth_bound_fps"], abs=0.05)
    assert synth.FRAMES_PER_SECOND / fps == pytest.approx(g["bandwidth_bound_rtf"], abs=0.005)
    assert fps / synth.FRAMES_PER_SECOND == pytest.approx(g["realtime_multiple"], abs=0.05)
    total = g["talker_gb_fp16"] + g["codepredictor_gb_fp16"] + g["codec_gb_fp16"]
    assert total == pytest.approx(g["total_gb_fp16"], abs=5e-4)


def test_algorithmic_frame_bytes_1p7b():
    s = synth.SHAPE_17B_KV32  # the fp32 Talker cache; the bf16 one below
    fb = bm.frame_bytes(s, 128)
    # Talker: 28 layers x (QKV 16.8 + o 8.4 + gate/up 50.3 + down 25.2 MB) + head 12.6 MB
    assert fb.talker_weights / 1e9 == pytest.approx(2.831, abs=0.001)
    # CodePredictor pass: 5 layers x 31.5 MB + head 4.2 MB + projection 4.2 MB
    assert fb.cp_pass_weights / 1e6 == pytest.approx(165.7, abs=0.1)
    # + Talker KV (28 layers x ~249 positions x 8 KB fp32 K+V) ~ 57 MB
    # + CodePredictor KV (fp32, 5 layers x 135 positions x 8 KB) ~ 5.5 MB
    run = bm.run_bytes(s, 128, 240) / 240
    assert run / 1e9 == pytest.approx(2.831 + 15 * 0.1657 + 0.0571 + 0.0055, abs=0.002)
    kv16 = bm.run_bytes(synth.SHAPE_17B, 128, 240) / 240
    assert (run - kv16) / 1e9 == pytest.approx(0.0286, abs=0.001)


def test_algorithmic_frame_bytes_0p6b():
    s = synth.SHAPE_06B
    fb = bm.frame_bytes(s, 64)
    assert fb.cp_pass_weights / 1e6 == pytest.approx(161.5, abs=0.1)
    # Talker 0.887 GB + 15 passes + bf16 Talker KV (~184 positions) + fp32 CodePredictor KV
    run = bm.run_bytes(s, 64, 240) / 240
    assert run / 1e9 == pytest.approx(0.887 + 15 * 0.1615 + 0.0423 / 2 + 0.0055, abs=0.002)


def test_talker_module_below_page_figure():
    """The page's Talker (3.483 GB) also holds a text embedding the shapes do not
    size; our counted Talker must stay below it."""
    t = bm.module_bytes(synth.SHAPE_17B)["talker"] / 1e9
    assert 2.8 < t < golden()["talker_gb_fp16"]


def test_fp8_frame_bytes_are_codes_plus_row_scales():
    """FP8 matrices cost one byte per weight plus an fp32 scale per output row
    (the row scales of the E4M3 format this library reads); gains, embedding rows
    and the KV cache are priced as in the bf16 shape."""
    s = synth.SHAPE_17B
    b = bm.frame_bytes(s, 200)
    f = bm.frame_bytes(synth.SHAPE_17B_FP8, 200)
    hq = s.n_q_heads * s.head_dim

    def mats(D, F, L, V):  # (rows, cols) of a stack's matrices and its head
        return [(s.qkv_rows, D), (D, hq), (2 * F, D), (D, F)] * L + [(V, D)]

    talker = mats(s.talker_hidden, s.talker_ffn, s.talker_layers, s.codec_vocab)
    cp = mats(s.cp_hidden, s.cp_ffn, s.cp_layers, s.cp_vocab) + [(s.cp_hidden, s.talker_hidden)]

    def fp8_minus_bf16(m):
        return sum(r * c + 4 * r - 2 * r * c for r, c in m)

    assert f.talker_weights - b.talker_weights == fp8_minus_bf16(talker)
    assert f.cp_pass_weights - b.cp_pass_weights == fp8_minus_bf16(cp)
    assert (f.embed_rows, f.kv_read, f.kv_write) == (b.embed_rows, b.kv_read, b.kv_write)
    # weights per frame: 2.66 GB in FP8 against 5.32 GB in bf16
    assert (f.talker_weights + 15 * f.cp_pass_weights) / 1e9 == pytest.approx(2.66, abs=0.01)
    assert (b.talker_weights + 15 * b.cp_pass_weights) / 1e9 == pytest.approx(5.32, abs=0.01)
