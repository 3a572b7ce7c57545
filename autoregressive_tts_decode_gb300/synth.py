"""Seeded synthetic inputs: model shapes, random weights, prompts, uniforms.

This module is the only code shared by the CUDA path and the CPU oracle.  It
holds none of the model's arithmetic: it describes the five workloads (layer
counts, widths, sampling settings) and draws the random numbers both sides
consume -- weight tensors in the library's row-major ``[out, in]`` layout,
prompt embeddings, ragged prompt lengths and the per-draw uniforms the sampler
turns into codes.

Sources for the shapes and settings:
  * "Running Qwen3-TTS on an AMD R9700" (flynnbody.com), section "Running
    Qwen3-TTS": 16 codebook tokens per 80 ms frame (1,920 samples at 24 kHz),
    the Talker producing the semantic token and the CodePredictor the other 15.
  * "qwen3-tts-hip" README (github.com/piedshag/qwen3-tts-hip), section
    "Library Usage": ``GenerateOptions`` sampling values (top_k 50, top_p 1.0,
    temperature 0.9, repetition_penalty 1.05 for the semantic token; the same
    without a repetition penalty for the sub-talker), ``max_frames`` 240 and
    ``EngineOptions::max_cache_steps``.
  * The workload list the benchmark runs (tiny, 0.6B-class, 1.7B-class,
    batched-16 and serving-128), which fixes layer counts, widths, heads,
    vocabularies, N(0, 0.02) weights and N(0, 1) prompts.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np

# Seeds of the synthetic workloads (weights, prompts, uniforms, prompt lengths).
SEED_WEIGHTS = 1234
SEED_PROMPTS = 1235
SEED_UNIFORMS = 1236
SEED_LENGTHS = 1237

N_CODEBOOKS = 16          # semantic token + 15 acoustic tokens per frame
SAMPLES_PER_FRAME = 1920  # 80 ms at 24 kHz
SAMPLE_RATE = 24000
FRAMES_PER_SECOND = SAMPLE_RATE / SAMPLES_PER_FRAME  # 12.5: real time

DTYPE_F32 = 0
DTYPE_BF16 = 1
DTYPE_FP8 = 2  # matrices as FP8 E4M3 codes with per-row fp32 scales; gains, embeddings bf16
FP8_MAX = 448.0  # largest finite E4M3 value


@dataclass(frozen=True)
class Sampling:
    """Per-stream sampling controls, mirroring ``GenerateOptions``.

    Semantic (Talker) token: do_sample, top_k, top_p, temperature,
    repetition_penalty.  Acoustic (CodePredictor, "sub-talker") tokens:
    sub_do_sample, sub_top_k, sub_top_p, sub_temperature -- the README lists
    no repetition penalty for them.
    """
    do_sample: bool = False
    top_k: int = 50
    top_p: float = 1.0
    temperature: float = 0.9
    repetition_penalty: float = 1.0
    sub_do_sample: bool = False
    sub_top_k: int = 50
    sub_top_p: float = 1.0
    sub_temperature: float = 0.9
    # stop conditions: the semantic code that ends a stream (< 0: none), and
    # the first special semantic code (codes >= it, other than eos_token, are
    # never drawn; <= 0: none)
    eos_token: int = -1
    special_from: int = 0


GREEDY = Sampling()
QWEN_DEFAULT_SAMPLING = Sampling(do_sample=True, top_k=50, top_p=1.0, temperature=0.9,
                                 repetition_penalty=1.05, sub_do_sample=True, sub_top_k=50,
                                 sub_top_p=1.0, sub_temperature=0.9)


@dataclass(frozen=True)
class ModelShape:
    talker_layers: int
    talker_hidden: int
    talker_ffn: int
    cp_layers: int
    cp_hidden: int
    cp_ffn: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    codec_vocab: int      # V_t, Talker codec vocabulary
    cp_vocab: int         # V_c, CodePredictor vocabulary per codebook
    weight_dtype: int     # DTYPE_F32, DTYPE_BF16 or DTYPE_FP8
    kv_dtype: int
    rms_eps: float = 1e-6
    rope_theta: float = 1e6
    qk_norm: int = 1
    n_codebooks: int = N_CODEBOOKS

    @property
    def has_proj(self) -> bool:
        return self.talker_hidden != self.cp_hidden

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim


@dataclass(frozen=True)
class Workload:
    name: str
    shape: ModelShape
    streams: int
    frames: int
    kv_cap: int
    page_size: int
    sampling: Sampling
    prompt_len: Optional[int] = None          # fixed length, or
    prompt_len_range: Optional[tuple] = None  # inclusive (lo, hi) drawn per stream

    def prompt_lengths(self, seed: int = SEED_LENGTHS) -> List[int]:
        if self.prompt_len is not None:
            return [self.prompt_len] * self.streams
        lo, hi = self.prompt_len_range
        rng = np.random.default_rng(seed)
        return [int(v) for v in rng.integers(lo, hi + 1, size=self.streams)]


TINY_SHAPE = ModelShape(talker_layers=2, talker_hidden=256, talker_ffn=768, cp_layers=1,
                        cp_hidden=256, cp_ffn=768, n_q_heads=4, n_kv_heads=2, head_dim=64,
                        codec_vocab=3072, cp_vocab=2048, weight_dtype=DTYPE_F32,
                        kv_dtype=DTYPE_F32)
# The 0.6B, 1.7B, batched and serving workloads keep bf16 weights and a bf16
# Talker KV cache (the oracle rounds its cached k, v to bf16 likewise); the
# CodePredictor cache is fp32.  SHAPE_17B_KV32 is the 1.7B shape with an fp32
# Talker cache, which the library also takes.
SHAPE_06B = ModelShape(talker_layers=28, talker_hidden=1024, talker_ffn=3072, cp_layers=5,
                       cp_hidden=1024, cp_ffn=3072, n_q_heads=16, n_kv_heads=8, head_dim=128,
                       codec_vocab=3072, cp_vocab=2048, weight_dtype=DTYPE_BF16,
                       kv_dtype=DTYPE_BF16)
SHAPE_17B = ModelShape(talker_layers=28, talker_hidden=2048, talker_ffn=6144, cp_layers=5,
                       cp_hidden=1024, cp_ffn=3072, n_q_heads=16, n_kv_heads=8, head_dim=128,
                       codec_vocab=3072, cp_vocab=2048, weight_dtype=DTYPE_BF16,
                       kv_dtype=DTYPE_BF16)
SHAPE_17B_KV16 = SHAPE_17B
SHAPE_17B_KV32 = dataclasses.replace(SHAPE_17B, kv_dtype=DTYPE_F32)
SHAPE_17B_FP8 = dataclasses.replace(SHAPE_17B, weight_dtype=DTYPE_FP8)

WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", TINY_SHAPE, streams=1, frames=8, kv_cap=64, page_size=16,
                     sampling=GREEDY, prompt_len=16),
    "0.6b": Workload("0.6b", SHAPE_06B, streams=1, frames=240, kv_cap=512, page_size=16,
                     sampling=GREEDY, prompt_len=64),
    "1.7b": Workload("1.7b", SHAPE_17B, streams=1, frames=240, kv_cap=512, page_size=16,
                     sampling=QWEN_DEFAULT_SAMPLING, prompt_len=128),
    "batched16": Workload("batched16", SHAPE_17B, streams=16, frames=240, kv_cap=512,
                          page_size=16, sampling=QWEN_DEFAULT_SAMPLING,
                          prompt_len_range=(32, 256)),
    "serving128": Workload("serving128", SHAPE_17B_KV16, streams=128, frames=64, kv_cap=2112,
                           page_size=16, sampling=GREEDY, prompt_len_range=(256, 2048)),
    # the 1.7B workload with 8-bit weight streaming (not one of the benchmark's
    # headline configurations: its own tolerance contract, see the tests)
    "1.7b-fp8": Workload("1.7b-fp8", SHAPE_17B_FP8, streams=1, frames=240, kv_cap=512, page_size=16,
                         sampling=QWEN_DEFAULT_SAMPLING, prompt_len=128),
}


def with_shape(w: Workload, **kw) -> Workload:
    """A copy of a workload with some ModelShape fields replaced (test helper)."""
    return dataclasses.replace(w, shape=dataclasses.replace(w.shape, **kw))


# --------------------------------------------------------------------------
# Weight tensors.  Names and layouts (all row-major [out, in]):
#   per layer: w_qkv [(Hq+2Hkv)*hd, D]  (q rows, then k rows, then v rows)
#              w_o   [D, Hq*hd]
#              w_gateup [2F, D]          (gate rows, then up rows)
#              w_down [D, F]
#              g_attn_norm [D], g_ffn_norm [D], g_q_norm [hd], g_k_norm [hd]
#   talker: g_final [D_t], w_head [V_t, D_t], e_codec [V_t, D_t]
#   code predictor: g_final [D_c], heads [15, V_c, D_c],
#                   embeds [15, V_c, D_t], w_proj [D_c, D_t] (only if D_t != D_c)
# --------------------------------------------------------------------------
LAYER_KEYS = ("w_qkv", "w_o", "w_gateup", "w_down",
              "g_attn_norm", "g_ffn_norm", "g_q_norm", "g_k_norm")
# per-output-row scales of the FP8 matrices (FP8 weights only)
LAYER_SCALE_KEYS = ("s_qkv", "s_o", "s_gateup", "s_down")
SCALE_OF = {"w_qkv": "s_qkv", "w_o": "s_o", "w_gateup": "s_gateup", "w_down": "s_down",
            "w_head": "s_head", "heads": "s_heads", "w_proj": "s_proj"}


def layer_shapes(s: ModelShape, hidden: int, ffn: int):
    return {
        "w_qkv": (s.qkv_rows, hidden),
        "w_o": (hidden, s.n_q_heads * s.head_dim),
        "w_gateup": (2 * ffn, hidden),
        "w_down": (hidden, ffn),
        "g_attn_norm": (hidden,),
        "g_ffn_norm": (hidden,),
        "g_q_norm": (s.head_dim,),
        "g_k_norm": (s.head_dim,),
    }


def weight_specs(s: ModelShape):
    """Ordered (name, shape, kind) list; kind 'mat' ~ N(0, 0.02), 'gain' = 1."""
    out = []
    for li in range(s.talker_layers):
        for k, shp in layer_shapes(s, s.talker_hidden, s.talker_ffn).items():
            out.append((f"talker.{li}.{k}", shp, "gain" if k.startswith("g_") else "mat"))
    out.append(("talker.g_final", (s.talker_hidden,), "gain"))
    out.append(("talker.w_head", (s.codec_vocab, s.talker_hidden), "mat"))
    out.append(("talker.e_codec", (s.codec_vocab, s.talker_hidden), "mat"))
    for li in range(s.cp_layers):
        for k, shp in layer_shapes(s, s.cp_hidden, s.cp_ffn).items():
            out.append((f"cp.{li}.{k}", shp, "gain" if k.startswith("g_") else "mat"))
    out.append(("cp.g_final", (s.cp_hidden,), "gain"))
    out.append(("cp.heads", (s.n_codebooks - 1, s.cp_vocab, s.cp_hidden), "mat"))
    out.append(("cp.embeds", (s.n_codebooks - 1, s.cp_vocab, s.talker_hidden), "mat"))
    if s.has_proj:
        out.append(("cp.w_proj", (s.cp_hidden, s.talker_hidden), "mat"))
    return out


def make_weights(s: ModelShape, seed: int = SEED_WEIGHTS, device="cpu", std: float = 0.02):
    """Random weights of the given shape: matrices N(0, std) drawn in fp32 from a
    torch generator seeded once and walked in ``weight_specs`` order, then rounded
    to the storage dtype (bf16 round-to-nearest-even); norm gains are 1.0.

    FP8 weights: the same fp32 draws; each matrix row r (the last dimension is
    the row) gets the scale s_r = max|w_r| / 448 (fp32) and the codes
    float8_e4m3fn(w / s_r) (torch's round-to-nearest-even), stored as uint8
    bytes under the matrix's name, the scales under its scale name (SCALE_OF);
    embedding tables and gains are bf16.

    The values depend on (seed, device type) only.
    """
    import torch
    fp8 = s.weight_dtype == DTYPE_FP8
    dt = torch.float32 if s.weight_dtype == DTYPE_F32 else torch.bfloat16
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    out = {}
    for name, shp, kind in weight_specs(s):
        if kind == "gain":
            out[name] = torch.ones(shp, dtype=dt, device=device)
            continue
        t = torch.empty(shp, dtype=torch.float32, device=device)
        t.normal_(0.0, std, generator=gen)
        short = name.rsplit(".", 1)[1]
        if fp8 and short in SCALE_OF:
            sc = (t.abs().amax(dim=-1) / FP8_MAX).to(torch.float32)
            q = (t / sc.unsqueeze(-1)).to(torch.float8_e4m3fn)
            out[name] = q.view(torch.uint8).contiguous()
            out[name.rsplit(".", 1)[0] + "." + SCALE_OF[short]] = sc.contiguous()
        else:
            out[name] = t.to(dt)
    return out


def make_prompts(s: ModelShape, lengths: List[int], seed: int = SEED_PROMPTS, device="cpu"):
    """One fp32 [len, D_t] prompt of N(0, 1) vectors per stream (drawn in stream order)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    out = []
    for n in lengths:
        t = torch.empty((n, s.talker_hidden), dtype=torch.float32, device=device)
        t.normal_(0.0, 1.0, generator=gen)
        out.append(t)
    return out


_M64 = np.uint64(0xFFFFFFFFFFFFFFFF)


def _splitmix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser (Steele, Lea and Flood, OOPSLA 2014), vectorised."""
    with np.errstate(over="ignore"):
        z = (z + np.uint64(0x9E3779B97F4A7C15)) & _M64
        z = ((z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)) & _M64
        z = ((z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)) & _M64
        return z ^ (z >> np.uint64(31))


def uniforms(stream_ids, frames: int, seed: int = SEED_UNIFORMS, frame0: int = 0) -> np.ndarray:
    """Counter-based uniforms u[stream, frame, codebook] in [0, 1), float32.

    u = (splitmix64(seed XOR (stream << 40 | frame << 8 | codebook)) >> 40) * 2**-24,
    i.e. 24 random bits, exact in fp32.  Shape [len(stream_ids), frames, 16].
    """
    s = np.asarray(stream_ids, dtype=np.uint64)[:, None, None]
    f = (np.arange(frames, dtype=np.uint64) + np.uint64(frame0))[None, :, None]
    c = np.arange(N_CODEBOOKS, dtype=np.uint64)[None, None, :]
    key = np.uint64(seed) ^ ((s << np.uint64(40)) | (f << np.uint64(8)) | c)
    bits = _splitmix64(key) >> np.uint64(40)
    return (bits.astype(np.float64) * 2.0 ** -24).astype(np.float32)
