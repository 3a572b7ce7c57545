"""ctypes front end of the CPU oracle (``q3oracle.c``).

Test infrastructure only: the tests, the package smoke check and the
benchmark's CPU-baseline leg use it; the CUDA library never does.  Weights are
handed over as CPU torch tensors (fp32 or bf16, row-major ``[out, in]``) whose
bytes the C code widens to double.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from typing import Dict, Optional, Sequence

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "q3oracle.c")
LIB = os.path.join(HERE, "libq3oracle.so")

LAYER_KEYS = ("w_qkv", "w_o", "w_gateup", "w_down",
              "g_attn_norm", "g_ffn_norm", "g_q_norm", "g_k_norm")


def build_cmd(out=None):
    # -ffp-contract=off: the sampler's float steps must not be fused.
    return ["gcc", "-O3", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
            SRC, "-o", out or LIB, "-lm"]


def build(force: bool = False) -> str:
    """Compiles the oracle library unless it is newer than its source; the
    result replaces the old file in one step (a process loading it meanwhile
    sees the old or the new library, never a partial one)."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = "%s.%d.tmp" % (LIB, os.getpid())
        subprocess.run(build_cmd(tmp), check=True)
        os.replace(tmp, LIB)
    return LIB


class _Cfg(C.Structure):
    _fields_ = [(n, C.c_int) for n in (
        "talker_layers", "talker_hidden", "talker_ffn", "cp_layers", "cp_hidden", "cp_ffn",
        "n_q_heads", "n_kv_heads", "head_dim", "codec_vocab", "cp_vocab", "n_codebooks",
        "kv_cap", "weight_dtype", "n_streams", "qk_norm", "kv_bf16")] + [
        ("rms_eps", C.c_double), ("rope_theta", C.c_double)]


class _Weights(C.Structure):
    _fields_ = [("talker_layers", C.POINTER(C.c_void_p)), ("talker_g_final", C.c_void_p),
                ("talker_w_head", C.c_void_p), ("talker_e_codec", C.c_void_p),
                ("cp_layers", C.POINTER(C.c_void_p)), ("cp_g_final", C.c_void_p),
                ("cp_heads", C.c_void_p), ("cp_embeds", C.c_void_p), ("cp_w_proj", C.c_void_p),
                ("s_head", C.c_void_p), ("s_cp_heads", C.c_void_p), ("s_cp_proj", C.c_void_p)]

# per-layer pointers: the LAYER_KEYS tensors, then the FP8 matrices' scales
LAYER_SCALES = ("s_qkv", "s_o", "s_gateup", "s_down")
NPTR = len(LAYER_KEYS) + len(LAYER_SCALES)


class _Sampling(C.Structure):
    _fields_ = [("do_sample", C.c_int), ("top_k", C.c_int), ("top_p", C.c_float),
                ("temperature", C.c_float), ("repetition_penalty", C.c_float),
                ("sub_do_sample", C.c_int), ("sub_top_k", C.c_int), ("sub_top_p", C.c_float),
                ("sub_temperature", C.c_float), ("eos_token", C.c_int), ("special_from", C.c_int)]


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(LIB)
        dp = C.POINTER(C.c_double)
        fp = C.POINTER(C.c_float)
        ip = C.POINTER(C.c_int)
        L.q3o_create.restype = C.c_void_p
        L.q3o_create.argtypes = [C.POINTER(_Cfg), C.POINTER(_Weights)]
        L.q3o_destroy.argtypes = [C.c_void_p]
        L.q3o_prefill.argtypes = [C.c_void_p, C.c_int, fp, C.c_int]
        L.q3o_pending.argtypes = [C.c_void_p, C.c_int, dp, dp]
        L.q3o_length.argtypes = [C.c_void_p, C.c_int]
        L.q3o_step_frame.argtypes = [C.c_void_p, C.c_int, C.POINTER(_Sampling), fp, ip, ip, fp]
        L.q3o_sample.argtypes = [fp, C.c_int, C.c_int, C.c_int, C.c_float, C.c_float, C.c_float,
                                 C.c_char_p, C.c_float, C.c_int, C.c_int]
        L.q3o_sample_f64.argtypes = [fp, C.c_int, C.c_int, C.c_int, C.c_double, C.c_double,
                                     C.c_double, C.c_char_p, C.c_double, dp, C.c_int, C.c_int]
        L.q3o_fp8_value.restype = C.c_double
        L.q3o_fp8_value.argtypes = [C.c_uint]
        L.q3o_expf.restype = C.c_float
        L.q3o_expf.argtypes = [C.c_float]
        L.q3o_rmsnorm.argtypes = [dp, C.c_int, fp, C.c_double, dp]
        L.q3o_rope.argtypes = [dp, C.c_int, C.c_int, C.c_double]
        L.q3o_attention.argtypes = [dp, dp, dp, C.c_int, C.c_int, C.c_int, C.c_int, dp]
        L.q3o_talker_stack.argtypes = [C.c_void_p, C.c_int, dp, C.c_int, C.c_int]
        L.q3o_max_threads.restype = C.c_int
        L.q3o_set_threads.argtypes = [C.c_int]
        L.q3o_cp_full.argtypes = [C.c_void_p, dp, fp]
        _lib = L
    return _lib


def _dptr(a: np.ndarray):
    return a.ctypes.data_as(C.POINTER(C.c_double))


def _fptr(a: np.ndarray):
    return a.ctypes.data_as(C.POINTER(C.c_float))


def _iptr(a: np.ndarray):
    return a.ctypes.data_as(C.POINTER(C.c_int))


def sampling_struct(sp) -> _Sampling:
    return _Sampling(int(sp.do_sample), int(sp.top_k), float(sp.top_p), float(sp.temperature),
                     float(sp.repetition_penalty), int(sp.sub_do_sample), int(sp.sub_top_k),
                     float(sp.sub_top_p), float(sp.sub_temperature),
                     int(getattr(sp, "eos_token", -1)), int(getattr(sp, "special_from", 0)))


def max_threads() -> int:
    return int(lib().q3o_max_threads())


def set_threads(n: int) -> None:
    """Thread count of the oracle's later parallel regions."""
    lib().q3o_set_threads(int(n))


def sample(logits: np.ndarray, do_sample: bool, top_k: int, top_p: float, temperature: float,
           rep_penalty: float = 1.0, history: Optional[np.ndarray] = None, u: float = 0.0,
           special_from: int = 0, eos_token: int = -1) -> int:
    """The float rule; ids >= special_from (when > 0) other than eos_token are
    never drawn."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    hist = None if history is None else np.ascontiguousarray(history, dtype=np.uint8).tobytes()
    return int(lib().q3o_sample(_fptr(lg), lg.size, int(do_sample), int(top_k), float(top_p),
                                float(temperature), float(rep_penalty), hist, float(u),
                                int(special_from), int(eos_token)))


def sample_f64(logits, do_sample, top_k, top_p, temperature, rep_penalty=1.0, history=None, u=0.0,
               special_from=0, eos_token=-1):
    """Returns (pick, margin): margin = distance of u*Z to the nearest CDF boundary / Z."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    hist = None if history is None else np.ascontiguousarray(history, dtype=np.uint8).tobytes()
    mg = C.c_double(0.0)
    pick = lib().q3o_sample_f64(_fptr(lg), lg.size, int(do_sample), int(top_k), float(top_p),
                                float(temperature), float(rep_penalty), hist, float(u), C.byref(mg),
                                int(special_from), int(eos_token))
    return int(pick), float(mg.value)


def fp8_value(code: int) -> float:
    """The value of an FP8 E4M3 code (the oracle's decoder)."""
    return float(lib().q3o_fp8_value(int(code)))


def expf(x: float) -> float:
    return float(lib().q3o_expf(float(x)))


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    g = np.ascontiguousarray(g, dtype=np.float32)
    y = np.empty_like(x)
    lib().q3o_rmsnorm(_dptr(x), x.size, _fptr(g), float(eps), _dptr(y))
    return y


def rope(v: np.ndarray, pos: int, theta: float) -> np.ndarray:
    v = np.array(v, dtype=np.float64, copy=True)
    lib().q3o_rope(_dptr(v), v.size, int(pos), float(theta))
    return v


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray) -> np.ndarray:
    """q [Hq, hd], K/V [S, Hkv, hd] -> o [Hq, hd] (single query over S positions)."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    K = np.ascontiguousarray(K, dtype=np.float64)
    V = np.ascontiguousarray(V, dtype=np.float64)
    Hq, hd = q.shape
    S, Hkv, _ = K.shape
    o = np.empty_like(q)
    lib().q3o_attention(_dptr(q), _dptr(K), _dptr(V), S, Hq, Hkv, hd, _dptr(o))
    return o


# The model shapes' code for a bf16 tensor (their weight_dtype / kv_dtype fields).
DTYPE_BF16_KV = 1


class Oracle:
    """The oracle model over CPU weight tensors (fp32 or bf16 torch tensors)."""

    def __init__(self, shape, weights: Dict[str, "object"], n_streams: int, kv_cap: int,
                 kv_bf16: Optional[bool] = None):
        """kv_bf16: the Talker KV cache holds bf16 values (each cached k, v is
        rounded to fp32 and then to the nearest bf16), as in a configuration
        whose cache is bf16.  None: as the shape's kv_dtype says."""
        if kv_bf16 is None:
            kv_bf16 = shape.kv_dtype == DTYPE_BF16_KV
        L = lib()
        self.shape = shape
        self.n_streams = n_streams
        self.kv_cap = kv_cap
        self._keep = {}
        for k, t in weights.items():
            t = t.detach().to("cpu").contiguous()
            self._keep[k] = t

        def p(name):
            t = self._keep.get(name)
            return None if t is None else C.c_void_p(t.data_ptr())

        def layer_ptrs(prefix, n):
            arr = (C.c_void_p * (n * NPTR))()
            for li in range(n):
                for j, k in enumerate(LAYER_KEYS + LAYER_SCALES):
                    t = self._keep.get(f"{prefix}.{li}.{k}")
                    arr[li * NPTR + j] = None if t is None else t.data_ptr()
            return arr

        tl = layer_ptrs("talker", shape.talker_layers)
        cl = layer_ptrs("cp", shape.cp_layers)
        self._tl, self._cl = tl, cl
        self._w = _Weights(C.cast(tl, C.POINTER(C.c_void_p)), p("talker.g_final"),
                           p("talker.w_head"), p("talker.e_codec"),
                           C.cast(cl, C.POINTER(C.c_void_p)), p("cp.g_final"), p("cp.heads"),
                           p("cp.embeds"), p("cp.w_proj"), p("talker.s_head"), p("cp.s_heads"),
                           p("cp.s_proj"))
        s = shape
        self._c = _Cfg(s.talker_layers, s.talker_hidden, s.talker_ffn, s.cp_layers, s.cp_hidden,
                       s.cp_ffn, s.n_q_heads, s.n_kv_heads, s.head_dim, s.codec_vocab, s.cp_vocab,
                       s.n_codebooks, kv_cap, s.weight_dtype, n_streams, s.qk_norm,
                       1 if kv_bf16 else 0, float(s.rms_eps), float(s.rope_theta))
        self._h = L.q3o_create(C.byref(self._c), C.byref(self._w))

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib().q3o_destroy(h)
            self._h = None

    def prefill(self, stream: int, embeds) -> None:
        e = np.ascontiguousarray(np.asarray(embeds, dtype=np.float32))
        rc = lib().q3o_prefill(self._h, stream, _fptr(e), e.shape[0])
        if rc != 0:
            raise ValueError(f"oracle prefill rejected (stream {stream}, len {e.shape[0]})")

    def pending(self, stream: int = 0):
        h = np.empty(self.shape.talker_hidden, dtype=np.float64)
        lg = np.empty(self.shape.codec_vocab, dtype=np.float64)
        lib().q3o_pending(self._h, stream, _dptr(h), _dptr(lg))
        return h, lg

    def length(self, stream: int = 0) -> int:
        return int(lib().q3o_length(self._h, stream))

    def step_frame(self, stream: int, sampling, u: Sequence[float], forced=None,
                   want_logits: bool = False):
        """Returns (codes int32[16], logits float32[V_t + 15 V_c] or None).  With
        sampling.eos_token >= 0, a frame whose fed semantic code is that code
        ends the stream (codes 1..15 are -1); every later frame of the stream
        yields sixteen -1 until the stream is prefilled again."""
        s = self.shape
        uu = np.ascontiguousarray(np.asarray(u, dtype=np.float32).reshape(16))
        codes = np.zeros(16, dtype=np.int32)
        fp = None
        if forced is not None:
            fa = np.ascontiguousarray(np.asarray(forced, dtype=np.int32).reshape(16))
            fp = _iptr(fa)
        lg = None
        lp = None
        if want_logits:
            lg = np.zeros(s.codec_vocab + 15 * s.cp_vocab, dtype=np.float32)
            lp = _fptr(lg)
        sp = sampling_struct(sampling)
        rc = lib().q3o_step_frame(self._h, stream, C.byref(sp), _fptr(uu), fp, _iptr(codes), lp)
        if rc != 0:
            raise ValueError("oracle KV cache full")
        return codes, lg

    def talker_stack(self, stream: int, x: np.ndarray, pos0: int) -> np.ndarray:
        x = np.array(x, dtype=np.float64, copy=True)
        lib().q3o_talker_stack(self._h, stream, _dptr(x), x.shape[0], pos0)
        return x

    def cp_full(self, tokens: np.ndarray) -> np.ndarray:
        """tokens [16, D_t] -> float32 logits [15, V_c] (one causal CodePredictor pass)."""
        t = np.ascontiguousarray(tokens, dtype=np.float64)
        out = np.zeros((15, self.shape.cp_vocab), dtype=np.float32)
        lib().q3o_cp_full(self._h, _dptr(t), _fptr(out))
        return out
