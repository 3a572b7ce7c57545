"""Algorithmic HBM bytes of one frame decode, for roofline accounting.

"Running Qwen3-TTS on an AMD R9700" (flynnbody.com), section "Running
Qwen3-TTS", models a frame's cost as the weight bytes read: the Talker once plus
the CodePredictor fifteen times.  This module counts the same thing from the
layer shapes, per frame and per stream position, as the bytes a frame must move
at least once: every weight matrix the step uses (once per use), the embedding
rows it looks up, the KV cache it reads and the KV it appends.

The page's own closed form counts whole modules (text embedding, all 15 heads
and tables in every CodePredictor pass); ``module_bytes`` reproduces its module
sizes so the two can be quoted side by side.
"""
from __future__ import annotations

from dataclasses import dataclass

from .synth import DTYPE_F32, DTYPE_FP8, ModelShape, N_CODEBOOKS


def esize(dtype: int) -> int:
    """Bytes of a gain or embedding element (bf16 beside FP8 matrices)."""
    return 4 if dtype == DTYPE_F32 else 2


def mat_bytes(s: ModelShape, rows: int, cols: int) -> int:
    """A [rows, cols] weight matrix: FP8 codes plus one fp32 scale per row, else
    rows * cols elements of the weight dtype."""
    if s.weight_dtype == DTYPE_FP8:
        return rows * cols + 4 * rows
    return rows * cols * esize(s.weight_dtype)


def layer_bytes(s: ModelShape, hidden: int, ffn: int) -> int:
    """One decoder layer: QKV, o_proj, gate/up, down, and its four gains."""
    return (mat_bytes(s, s.qkv_rows, hidden) + mat_bytes(s, hidden, s.n_q_heads * s.head_dim)
            + mat_bytes(s, 2 * ffn, hidden) + mat_bytes(s, hidden, ffn)
            + (2 * hidden + 2 * s.head_dim) * esize(s.weight_dtype))


def layer_weight_elems(s: ModelShape, hidden: int, ffn: int) -> int:
    return (s.qkv_rows * hidden + hidden * s.n_q_heads * s.head_dim + 2 * ffn * hidden
            + hidden * ffn + 2 * hidden + 2 * s.head_dim)


@dataclass
class FrameBytes:
    talker_weights: int
    cp_pass_weights: int       # one CodePredictor pass (layers + final norm + one head + proj)
    embed_rows: int            # the 16 embedding rows of the next Talker input + 15 CP input rows
    kv_read: int               # Talker + CodePredictor KV read
    kv_write: int

    @property
    def total(self) -> int:
        return (self.talker_weights + (N_CODEBOOKS - 1) * self.cp_pass_weights + self.embed_rows
                + self.kv_read + self.kv_write)


def frame_bytes(s: ModelShape, talker_pos: int) -> FrameBytes:
    """Bytes for one frame of one stream whose Talker step writes position talker_pos."""
    e = esize(s.weight_dtype)
    kv_e = esize(s.kv_dtype)
    tw = (s.talker_layers * layer_bytes(s, s.talker_hidden, s.talker_ffn) + s.talker_hidden * e
          + mat_bytes(s, s.codec_vocab, s.talker_hidden))
    cw = (s.cp_layers * layer_bytes(s, s.cp_hidden, s.cp_ffn) + s.cp_hidden * e
          + mat_bytes(s, s.cp_vocab, s.cp_hidden))
    if s.has_proj:
        cw += mat_bytes(s, s.cp_hidden, s.talker_hidden)
    # next Talker input: 16 rows; CodePredictor inputs: E_t[c0] in pass 0 and
    # E_cp[j-1][c_j] in passes 1..14.
    emb = (N_CODEBOOKS + (N_CODEBOOKS - 1)) * s.talker_hidden * e
    kvh = s.n_kv_heads * s.head_dim
    # Talker: reads K and V of positions 0..talker_pos, writes one position.
    kv_read = s.talker_layers * (talker_pos + 1) * kvh * 2 * kv_e
    kv_write = s.talker_layers * kvh * 2 * kv_e
    # CodePredictor (fp32 cache): pass 0 covers positions 0,1; pass j reads 0..j+1.
    cp_reads = sum(j + 2 for j in range(N_CODEBOOKS - 1))
    kv_read += s.cp_layers * cp_reads * kvh * 2 * 4
    kv_write += s.cp_layers * N_CODEBOOKS * kvh * 2 * 4
    return FrameBytes(tw, cw, emb, kv_read, kv_write)


def run_bytes(s: ModelShape, prompt_len: int, frames: int) -> int:
    """Bytes of `frames` frames after a prompt of prompt_len (frame f writes position prompt_len+f)."""
    return sum(frame_bytes(s, prompt_len + f).total for f in range(frames))


def batched_step_bytes(s: ModelShape, positions) -> int:
    """One frame for each of several streams, weights shared: the weights once, KV per stream."""
    fb = [frame_bytes(s, p) for p in positions]
    w = fb[0].talker_weights + (N_CODEBOOKS - 1) * fb[0].cp_pass_weights
    return w + sum(f.embed_rows + f.kv_read + f.kv_write for f in fb)


def module_bytes(s: ModelShape) -> dict:
    """Whole-module sizes as the page counts them: Talker layers + final norm + codec
    head + codec embedding (no text embedding, which the shapes do not fix), and the
    CodePredictor with all 15 heads, all 15 embedding tables and the projection."""
    e = esize(s.weight_dtype)
    talker = (s.talker_layers * layer_weight_elems(s, s.talker_hidden, s.talker_ffn)
              + s.talker_hidden + 2 * s.codec_vocab * s.talker_hidden) * e
    cp = (s.cp_layers * layer_weight_elems(s, s.cp_hidden, s.cp_ffn) + s.cp_hidden
          + (N_CODEBOOKS - 1) * s.cp_vocab * (s.cp_hidden + s.talker_hidden)) * e
    if s.has_proj:
        cp += s.cp_hidden * s.talker_hidden * e
    return {"talker": talker, "code_predictor": cp}


def page_frame_bytes(talker_gb: float, cp_gb: float) -> float:
    """The page's closed form: bytes(Talker once) + 15 * bytes(CodePredictor once)."""
    return talker_gb + (N_CODEBOOKS - 1) * cp_gb
