"""ctypes binding of libq3tts (include/q3tts.h): argument marshalling only.

Every step of the decode runs in the CUDA library; this module turns torch
tensors into device pointers and status codes into exceptions.  It refuses to
work without the built library (no CPU path exists).
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Dict, Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libq3tts.so")

OK = 0
ERR_ARG, ERR_CAPACITY, ERR_CUDA, ERR_TIMEOUT, ERR_UNSUPPORTED, ERR_STATE = -1, -2, -3, -4, -5, -6
ERR_SCRATCH = -7
STATIC_SCRATCH_BYTES = 786432
F32, BF16, FP8 = 0, 1, 2
MAX_STREAMS = 256
N_CODEBOOKS = 16

LAYER_KEYS = ("w_qkv", "w_o", "w_gateup", "w_down",
              "g_attn_norm", "g_ffn_norm", "g_q_norm", "g_k_norm")
LAYER_SCALES = ("s_qkv", "s_o", "s_gateup", "s_down")  # FP8 matrices' per-row scales


class Q3TTSError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {strerror(code)} ({code})")
        self.code = code


class Config(C.Structure):
    _fields_ = [(n, C.c_int) for n in (
        "talker_layers", "talker_hidden", "talker_ffn", "cp_layers", "cp_hidden", "cp_ffn",
        "n_q_heads", "n_kv_heads", "head_dim", "codec_vocab", "cp_vocab", "n_codebooks",
        "max_streams", "kv_cap_steps", "page_size", "kv_pages", "prefill_chunk",
        "weight_dtype", "kv_dtype", "qk_norm")] + [("rms_eps", C.c_float), ("rope_theta", C.c_float)]


class LayerWeights(C.Structure):
    _fields_ = [(k, C.c_void_p) for k in LAYER_KEYS + LAYER_SCALES]


class Weights(C.Structure):
    _fields_ = [("talker_layers", C.POINTER(LayerWeights)), ("talker_g_final", C.c_void_p),
                ("talker_w_head", C.c_void_p), ("talker_e_codec", C.c_void_p),
                ("cp_layers", C.POINTER(LayerWeights)), ("cp_g_final", C.c_void_p),
                ("cp_heads", C.c_void_p), ("cp_embeds", C.c_void_p), ("cp_w_proj", C.c_void_p),
                ("s_head", C.c_void_p), ("s_cp_heads", C.c_void_p), ("s_cp_proj", C.c_void_p)]


class Sampling(C.Structure):
    _fields_ = [("do_sample", C.c_int), ("top_k", C.c_int), ("top_p", C.c_float),
                ("temperature", C.c_float), ("repetition_penalty", C.c_float),
                ("sub_do_sample", C.c_int), ("sub_top_k", C.c_int), ("sub_top_p", C.c_float),
                ("sub_temperature", C.c_float), ("eos_token", C.c_int), ("special_from", C.c_int)]


EXPORTS = ("q3tts_workspace_size", "q3tts_create", "q3tts_prefill", "q3tts_step_frame",
           "q3tts_read_pending", "q3tts_reset", "q3tts_stream_length", "q3tts_sync_status",
           "q3tts_kernel_launches", "q3tts_destroy", "q3tts_strerror",
           "q3tts_step_frame_static", "q3tts_debug_fail_barrier", "q3tts_stream_finished",
           "q3tts_step_frames", "q3tts_frames_ready")
MAX_CHUNK = 64

_lib = None


def load(path: str = LIB_PATH):
    """Loads libq3tts.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libq3tts.so is not built ({path}); run __graft_entry__.build()")
    L = C.CDLL(path)
    vp = C.c_void_p
    L.q3tts_workspace_size.restype = C.c_size_t
    L.q3tts_workspace_size.argtypes = [C.POINTER(Config)]
    L.q3tts_create.argtypes = [C.POINTER(Config), C.POINTER(Weights), vp, C.c_size_t, vp,
                               C.POINTER(vp)]
    L.q3tts_prefill.argtypes = [vp, C.c_int, vp, C.c_int]
    L.q3tts_step_frame.argtypes = [vp, C.POINTER(Sampling), C.POINTER(C.c_int32), C.c_int, vp, vp,
                                   vp, vp]
    L.q3tts_step_frame_static.argtypes = [vp, C.POINTER(Sampling), C.c_int, vp, vp, vp, vp]
    L.q3tts_read_pending.argtypes = [vp, C.c_int, vp, vp]
    L.q3tts_reset.argtypes = [vp, C.c_int]
    L.q3tts_stream_length.argtypes = [vp, C.c_int]
    L.q3tts_sync_status.argtypes = [vp]
    L.q3tts_destroy.argtypes = [vp]
    L.q3tts_kernel_launches.restype = C.c_uint64
    L.q3tts_kernel_launches.argtypes = [vp]
    L.q3tts_debug_fail_barrier.argtypes = [vp, C.c_int, C.c_int]
    L.q3tts_stream_finished.argtypes = [vp, C.c_int, C.POINTER(C.c_int)]
    L.q3tts_step_frames.argtypes = [vp, C.POINTER(Sampling), C.POINTER(C.c_int32), C.c_int, C.c_int, vp, vp,
                                    vp, vp]
    L.q3tts_frames_ready.argtypes = [vp]
    L.q3tts_strerror.restype = C.c_char_p
    L.q3tts_strerror.argtypes = [C.c_int]
    _lib = L
    return L


def strerror(code: int) -> str:
    try:
        return load().q3tts_strerror(code).decode()
    except RuntimeError:
        return f"error {code}"


def _check(rc: int, what: str):
    if rc != OK:
        raise Q3TTSError(rc, what)


def make_config(shape, max_streams: int, kv_cap: int, page_size: int = 16, kv_pages: int = 0,
                prefill_chunk: int = 0) -> Config:
    s = shape
    return Config(s.talker_layers, s.talker_hidden, s.talker_ffn, s.cp_layers, s.cp_hidden,
                  s.cp_ffn, s.n_q_heads, s.n_kv_heads, s.head_dim, s.codec_vocab, s.cp_vocab,
                  s.n_codebooks, max_streams, kv_cap, page_size, kv_pages, prefill_chunk,
                  s.weight_dtype, s.kv_dtype, s.qk_norm, float(s.rms_eps), float(s.rope_theta))


def sampling_struct(sp) -> Sampling:
    return Sampling(int(sp.do_sample), int(sp.top_k), float(sp.top_p), float(sp.temperature),
                    float(sp.repetition_penalty), int(sp.sub_do_sample), int(sp.sub_top_k),
                    float(sp.sub_top_p), float(sp.sub_temperature),
                    int(getattr(sp, "eos_token", -1)), int(getattr(sp, "special_from", 0)))


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need(t, name: str, dtype, numel: int, what: str):
    """Raises Q3TTSError(ERR_ARG) unless t is a contiguous CUDA tensor of the
    given dtype with at least numel elements (checked before the C call, so a
    wrong buffer is an error instead of an out-of-bounds device write)."""
    import torch
    ok = (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous() and t.dtype == dtype
          and t.numel() >= numel)
    if not ok:
        raise Q3TTSError(ERR_ARG, f"{what}: {name} must be a contiguous CUDA {dtype} tensor "
                                  f"of at least {numel} elements")


class Engine:
    """One libq3tts handle over device weights (dict of CUDA tensors named as in
    ``synth.weight_specs``) and a workspace allocated here through torch."""

    def __init__(self, shape, weights: Dict[str, "object"], max_streams: int, kv_cap: int,
                 page_size: int = 16, kv_pages: int = 0, prefill_chunk: int = 0, stream=None):
        import torch
        L = load()
        self.shape = shape
        self.max_streams = max_streams
        self.cfg = make_config(shape, max_streams, kv_cap, page_size, kv_pages, prefill_chunk)
        self._w = weights
        for k, t in weights.items():
            if not t.is_cuda or not t.is_contiguous():
                raise ValueError(f"weight {k} must be a contiguous CUDA tensor")
        def layer(prefix):
            return LayerWeights(*[_ptr(weights.get(f"{prefix}.{k}")) for k in LAYER_KEYS + LAYER_SCALES])

        tl = (LayerWeights * shape.talker_layers)()
        for i in range(shape.talker_layers):
            tl[i] = layer(f"talker.{i}")
        cl = (LayerWeights * shape.cp_layers)()
        for i in range(shape.cp_layers):
            cl[i] = layer(f"cp.{i}")
        proj = weights.get("cp.w_proj")
        self._tl, self._cl = tl, cl
        self.wstruct = Weights(tl, weights["talker.g_final"].data_ptr(),
                               weights["talker.w_head"].data_ptr(),
                               weights["talker.e_codec"].data_ptr(), cl,
                               weights["cp.g_final"].data_ptr(), weights["cp.heads"].data_ptr(),
                               weights["cp.embeds"].data_ptr(), _ptr(proj), _ptr(weights.get("talker.s_head")),
                               _ptr(weights.get("cp.s_heads")), _ptr(weights.get("cp.s_proj")))
        n = L.q3tts_workspace_size(C.byref(self.cfg))
        if n == 0:
            raise Q3TTSError(ERR_ARG, "q3tts_workspace_size")
        self.workspace_bytes = int(n)
        self.workspace = torch.empty(int(n), dtype=torch.uint8, device="cuda")
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        h = C.c_void_p()
        _check(L.q3tts_create(C.byref(self.cfg), C.byref(self.wstruct),
                              self.workspace.data_ptr(), n, C.c_void_p(self.stream.cuda_stream),
                              C.byref(h)), "q3tts_create")
        self.h = h

    def close(self):
        if getattr(self, "h", None) is not None and self.h.value:
            # queued work still reads the workspace this object owns: wait for
            # it (a recorded error was the caller's to collect) before release
            load().q3tts_sync_status(self.h)
            load().q3tts_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def prefill(self, stream_id: int, embeds) -> None:
        import torch
        if embeds.dim() != 2 or embeds.shape[1] != self.shape.talker_hidden:
            raise Q3TTSError(ERR_ARG, "q3tts_prefill: embeds must be [len, talker_hidden]")
        _need(embeds, "embeds", torch.float32, embeds.shape[0] * self.shape.talker_hidden,
              "q3tts_prefill")
        _check(load().q3tts_prefill(self.h, stream_id, embeds.data_ptr(), embeds.shape[0]),
               "q3tts_prefill")

    def step_frame(self, stream_ids: Sequence[int], sampling, uniforms, codes, forced=None,
                   logits=None) -> None:
        """uniforms: CUDA fp32 [n, 16]; codes: CUDA int32 [n, 16] (written);
        forced: None or CUDA int32 [n, 16]; logits: None or CUDA fp32
        [n, V_t + 15 V_c].  `sampling` is one Sampling-like object or a list."""
        n = len(stream_ids)
        self._check_frame_buffers(n, uniforms, codes, forced, logits, "q3tts_step_frame")
        if not isinstance(sampling, (list, tuple)):
            sampling = [sampling] * n
        sp = (Sampling * n)(*[sampling_struct(x) for x in sampling])
        ids = (C.c_int32 * n)(*[int(i) for i in stream_ids])
        _check(load().q3tts_step_frame(self.h, sp, ids, n, uniforms.data_ptr(), codes.data_ptr(),
                                       _ptr(forced), _ptr(logits)), "q3tts_step_frame")

    def step_frame_static(self, stream_id: int, sampling, uniforms, codes, forced=None,
                          logits=None) -> None:
        """One frame of one stream through q3tts_step_frame_static (scratch in the
        library's static device array); tensors as for step_frame with n = 1."""
        self._check_frame_buffers(1, uniforms, codes, forced, logits, "q3tts_step_frame_static")
        sp = sampling_struct(sampling)
        _check(load().q3tts_step_frame_static(self.h, C.byref(sp), int(stream_id),
                                              uniforms.data_ptr(), codes.data_ptr(),
                                              _ptr(forced), _ptr(logits)),
               "q3tts_step_frame_static")

    def step_frames(self, stream_ids: Sequence[int], sampling, uniforms, codes, codes_host=None,
                    forced=None) -> None:
        """q3tts_step_frames: F = uniforms.shape[0] frames (<= MAX_CHUNK) enqueued back
        to back.  uniforms: CUDA fp32 [F, n, 16]; codes: CUDA int32 [F, n, 16]
        (written); codes_host: None or a pinned CPU int32 [F, n, 16] tensor (written
        asynchronously, frame by frame); forced: None or CUDA int32 [F, n, 16]."""
        import torch
        n = len(stream_ids)
        F = int(uniforms.shape[0])
        what = "q3tts_step_frames"
        _need(uniforms, "uniforms", torch.float32, F * n * N_CODEBOOKS, what)
        _need(codes, "codes", torch.int32, F * n * N_CODEBOOKS, what)
        if forced is not None:
            _need(forced, "forced", torch.int32, F * n * N_CODEBOOKS, what)
        hp = None
        if codes_host is not None:
            ok = (isinstance(codes_host, torch.Tensor) and not codes_host.is_cuda and codes_host.is_contiguous()
                  and codes_host.dtype == torch.int32 and codes_host.numel() >= F * n * N_CODEBOOKS)
            if not ok:
                raise Q3TTSError(ERR_ARG, f"{what}: codes_host must be a contiguous CPU int32 tensor")
            hp = codes_host.data_ptr()
        if not isinstance(sampling, (list, tuple)):
            sampling = [sampling] * n
        sp = (Sampling * n)(*[sampling_struct(x) for x in sampling])
        ids = (C.c_int32 * n)(*[int(i) for i in stream_ids])
        _check(load().q3tts_step_frames(self.h, sp, ids, n, F, uniforms.data_ptr(), codes.data_ptr(), hp,
                                        _ptr(forced)), what)

    def frames_ready(self) -> int:
        """Frames of the latest step_frames chunk whose codes have landed (non-blocking)."""
        r = load().q3tts_frames_ready(self.h)
        if r < 0:
            _check(r, "q3tts_frames_ready")
        return r

    def stream_codes(self, stream_ids: Sequence[int], sampling, uniforms, chunk: int):
        """Frame-incremental decode of the given streams, chunk frames at a time
        (the counterpart of a streaming session's next_audio_chunk): yields numpy
        int32 arrays [frames, n, 16] of codes in order.  uniforms: CUDA fp32
        [total_frames, n, 16].  Double-buffered: chunk k + 1 is enqueued before
        the host waits for chunk k, so the GPU never idles on the host."""
        import numpy as np
        import torch
        n = len(stream_ids)
        total = int(uniforms.shape[0])
        chunk = max(1, min(int(chunk), MAX_CHUNK))
        dev = [torch.zeros((chunk, n, N_CODEBOOKS), dtype=torch.int32, device="cuda") for _ in range(2)]
        host = [torch.zeros((chunk, n, N_CODEBOOKS), dtype=torch.int32).pin_memory() for _ in range(2)]
        done = [torch.cuda.Event(), torch.cuda.Event()]
        spans = [(f0, min(total, f0 + chunk)) for f0 in range(0, total, chunk)]

        def submit(k):
            f0, f1 = spans[k]
            b = k & 1
            self.step_frames(stream_ids, sampling, uniforms[f0:f1].contiguous(), dev[b][:f1 - f0],
                             codes_host=host[b][:f1 - f0])
            done[b].record(self.stream)

        if spans:
            submit(0)
        for k in range(len(spans)):
            if k + 1 < len(spans):
                submit(k + 1)
            done[k & 1].synchronize()
            f0, f1 = spans[k]
            yield np.array(host[k & 1][:f1 - f0].numpy(), copy=True)

    def _check_frame_buffers(self, n, uniforms, codes, forced, logits, what):
        import torch
        _need(uniforms, "uniforms", torch.float32, n * N_CODEBOOKS, what)
        _need(codes, "codes", torch.int32, n * N_CODEBOOKS, what)
        if forced is not None:
            _need(forced, "forced", torch.int32, n * N_CODEBOOKS, what)
        if logits is not None:
            s = self.shape
            _need(logits, "logits", torch.float32, n * (s.codec_vocab + 15 * s.cp_vocab), what)

    def read_pending(self, stream_id: int):
        import torch
        hdn = torch.empty(self.shape.talker_hidden, dtype=torch.float32, device="cuda")
        lg = torch.empty(self.shape.codec_vocab, dtype=torch.float32, device="cuda")
        _check(load().q3tts_read_pending(self.h, stream_id, hdn.data_ptr(), lg.data_ptr()),
               "q3tts_read_pending")
        return hdn, lg

    def reset(self, stream_id: int = -1) -> None:
        _check(load().q3tts_reset(self.h, stream_id), "q3tts_reset")

    def length(self, stream_id: int) -> int:
        rc = load().q3tts_stream_length(self.h, stream_id)
        if rc < 0:
            raise Q3TTSError(rc, "q3tts_stream_length")
        return rc

    def finished(self, stream_id: int) -> bool:
        """Whether the stream fed its end-of-stream code since its last prefill
        (waits for the engine's stream)."""
        f = C.c_int(0)
        _check(load().q3tts_stream_finished(self.h, stream_id, C.byref(f)), "q3tts_stream_finished")
        return bool(f.value)

    def kernel_launches(self) -> int:
        return int(load().q3tts_kernel_launches(self.h))

    def debug_fail_barrier(self, barrier: int, wait_us: int) -> None:
        """Arms the next persistent frame to leave out CTA 0's arrival at grid
        barrier `barrier` with every wait bounded to wait_us (failure-path test)."""
        _check(load().q3tts_debug_fail_barrier(self.h, int(barrier), int(wait_us)),
               "q3tts_debug_fail_barrier")

    def sync(self) -> None:
        _check(load().q3tts_sync_status(self.h), "q3tts_sync_status")
