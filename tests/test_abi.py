"""The C ABI without a GPU: the library builds for sm_103a, loads, and exports
every function include/q3tts.h declares; the binding mirrors the header's
structs and constants; the host-side argument checks (NULL handles, unaligned
weights) answer before any device work; every status code has its text."""
import ctypes
import os
import re

import pytest

from autoregressive_tts_decode_gb300 import build, q3tts

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q3tts.h")


def header_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"\b(q3tts_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ctypes.CDLL(build.LIB)


def test_exports_every_declared_function(lib):
    names = header_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(q3tts.EXPORTS)


def test_header_constants_match_binding():
    src = open(HEADER).read()
    consts = dict(re.findall(r"#define (Q3TTS_[A-Z_0-9]+) \(?(-?\d+)\)?", src))
    assert int(consts["Q3TTS_ERR_ARG"]) == q3tts.ERR_ARG
    assert int(consts["Q3TTS_ERR_CAPACITY"]) == q3tts.ERR_CAPACITY
    assert int(consts["Q3TTS_ERR_CUDA"]) == q3tts.ERR_CUDA
    assert int(consts["Q3TTS_ERR_TIMEOUT"]) == q3tts.ERR_TIMEOUT
    assert int(consts["Q3TTS_ERR_UNSUPPORTED"]) == q3tts.ERR_UNSUPPORTED
    assert int(consts["Q3TTS_ERR_STATE"]) == q3tts.ERR_STATE
    assert int(consts["Q3TTS_ERR_SCRATCH"]) == q3tts.ERR_SCRATCH
    assert int(consts["Q3TTS_STATIC_SCRATCH_BYTES"]) == q3tts.STATIC_SCRATCH_BYTES
    assert int(consts["Q3TTS_MAX_STREAMS"]) == q3tts.MAX_STREAMS
    assert int(consts["Q3TTS_BF16"]) == q3tts.BF16


def test_struct_layouts_match_header():
    src = open(HEADER).read()

    def fields(struct):
        body = re.search(r"typedef struct " + struct + r" \{(.*?)\} " + struct, src, re.S).group(1)
        body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
        out = []
        for decl in body.split(";"):
            decl = decl.strip()
            if not decl:
                continue
            names = decl.split(None, 1)[1] if not decl.startswith("const") else decl.split("*", 1)[1]
            out += [n.strip().lstrip("*") for n in names.split(",")]
        return out

    assert fields("q3tts_config") == [f[0] for f in q3tts.Config._fields_]
    assert fields("q3tts_sampling") == [f[0] for f in q3tts.Sampling._fields_]
    assert fields("q3tts_layer_weights") == [f[0] for f in q3tts.LayerWeights._fields_]
    assert fields("q3tts_weights") == [f[0] for f in q3tts.Weights._fields_]


def test_workspace_size_without_gpu(lib):
    from autoregressive_tts_decode_gb300 import synth
    L = q3tts.load(build.LIB)
    cfg = q3tts.make_config(synth.TINY_SHAPE, 1, 64)
    n = L.q3tts_workspace_size(ctypes.byref(cfg))
    assert n > 0
    bad = q3tts.make_config(synth.TINY_SHAPE, 1, 64)
    bad.head_dim = 96
    assert L.q3tts_workspace_size(ctypes.byref(bad)) == 0
    assert L.q3tts_strerror(q3tts.ERR_CAPACITY).decode().startswith("KV cache")


def test_binding_refuses_missing_library(tmp_path):
    with pytest.raises(RuntimeError):
        q3tts._lib_saved = q3tts._lib
        try:
            q3tts._lib = None
            q3tts.load(str(tmp_path / "nope.so"))
        finally:
            q3tts._lib = q3tts._lib_saved


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    """No CPU fallback: without the built library the binding raises instead of
    running anything."""
    monkeypatch.setattr(q3tts, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        q3tts.load(str(tmp_path / "libq3tts.so"))


def _fake_weights(shape, base=1 << 40):
    """Weights struct of distinct, 256-byte aligned fake addresses (never
    dereferenced: the calls below must stop at their argument checks)."""
    addr = [base]

    def nxt():
        addr[0] += 1 << 20
        return addr[0]
    tl = (q3tts.LayerWeights * shape.talker_layers)()
    for i in range(shape.talker_layers):
        tl[i] = q3tts.LayerWeights(*[nxt() for _ in q3tts.LAYER_KEYS])
    cl = (q3tts.LayerWeights * shape.cp_layers)()
    for i in range(shape.cp_layers):
        cl[i] = q3tts.LayerWeights(*[nxt() for _ in q3tts.LAYER_KEYS])
    w = q3tts.Weights(tl, nxt(), nxt(), nxt(), cl, nxt(), nxt(), nxt(),
                      nxt() if shape.has_proj else None)
    return w, tl, cl


def test_create_rejects_unaligned_weight_pointers(lib):
    """Every weight and gain pointer must be 16-byte aligned (the kernels read
    them with 16-byte vector loads and bulk copies): an 8-byte offset in any one
    of them is Q3TTS_ERR_ARG, returned before anything touches the device."""
    import torch
    from autoregressive_tts_decode_gb300 import synth
    L = q3tts.load(build.LIB)
    shape = synth.SHAPE_17B
    cfg = q3tts.make_config(shape, 1, 512)
    ws = ctypes.c_void_p(1 << 41)
    top = ["talker_g_final", "talker_w_head", "talker_e_codec", "cp_g_final", "cp_heads",
           "cp_embeds", "cp_w_proj"]
    cases = [(None, f) for f in top] + [("talker", k) for k in q3tts.LAYER_KEYS] + \
            [("cp", k) for k in q3tts.LAYER_KEYS]
    for where, field in cases:
        w, tl, cl = _fake_weights(shape)
        if where is None:
            setattr(w, field, getattr(w, field) + 8)
        else:
            arr = tl if where == "talker" else cl
            setattr(arr[len(arr) - 1], field, getattr(arr[len(arr) - 1], field) + 8)
        h = ctypes.c_void_p()
        rc = L.q3tts_create(ctypes.byref(cfg), ctypes.byref(w), ws, 1 << 60, None, ctypes.byref(h))
        assert rc == q3tts.ERR_ARG, (where, field, rc)
        assert not h.value
    if not torch.cuda.is_available():
        # the aligned set passes the argument checks and stops at the first
        # CUDA call, which fails here for want of a device
        w, tl, cl = _fake_weights(shape)
        h = ctypes.c_void_p()
        rc = L.q3tts_create(ctypes.byref(cfg), ctypes.byref(w), ws, 1 << 60, None, ctypes.byref(h))
        assert rc == q3tts.ERR_CUDA


def test_every_call_rejects_a_null_handle_on_the_host(lib):
    """The calls' argument checks come before any device work: every function
    the header declares, given a NULL handle (or NULL required pointers),
    returns Q3TTS_ERR_ARG -- here, with no device at all.  kernel_launches(NULL)
    is 0, destroy(NULL) is a no-op and create clears its output handle."""
    L = q3tts.load(build.LIB)
    N, E = None, q3tts.ERR_ARG
    out = ctypes.c_void_p(0x1000)
    fin = ctypes.c_int(7)
    calls = {
        "q3tts_workspace_size": (lambda: L.q3tts_workspace_size(N), 0),
        "q3tts_create": (lambda: L.q3tts_create(N, N, N, 0, N, ctypes.byref(out)), E),
        "q3tts_prefill": (lambda: L.q3tts_prefill(N, 0, N, 1), E),
        "q3tts_step_frame": (lambda: L.q3tts_step_frame(N, N, N, 1, N, N, N, N), E),
        "q3tts_step_frames": (lambda: L.q3tts_step_frames(N, N, N, 1, 1, N, N, N, N), E),
        "q3tts_frames_ready": (lambda: L.q3tts_frames_ready(N), E),
        "q3tts_step_frame_static": (lambda: L.q3tts_step_frame_static(N, N, 0, N, N, N, N), E),
        "q3tts_read_pending": (lambda: L.q3tts_read_pending(N, 0, N, N), E),
        "q3tts_reset": (lambda: L.q3tts_reset(N, -1), E),
        "q3tts_stream_length": (lambda: L.q3tts_stream_length(N, 0), E),
        "q3tts_stream_finished": (lambda: L.q3tts_stream_finished(N, 0, ctypes.byref(fin)), E),
        "q3tts_sync_status": (lambda: L.q3tts_sync_status(N), E),
        "q3tts_kernel_launches": (lambda: L.q3tts_kernel_launches(N), 0),
        "q3tts_debug_fail_barrier": (lambda: L.q3tts_debug_fail_barrier(N, 0, 1000), E),
        "q3tts_destroy": (lambda: L.q3tts_destroy(N), ...),  # void: only returns
        "q3tts_strerror": (lambda: L.q3tts_strerror(q3tts.ERR_ARG), b"invalid argument"),
    }
    assert set(calls) == set(header_functions())
    for name, (call, want) in calls.items():
        got = call()
        assert want is ... or got == want, name
    assert out.value is None
    assert fin.value == 7


def test_strerror_describes_every_status_code(lib):
    """Each status code the header defines has its own description; any other
    value reads "unknown error" (a static string, never NULL)."""
    L = q3tts.load(build.LIB)
    src = open(HEADER).read()
    codes = {k: int(v) for k, v in re.findall(r"#define (Q3TTS_(?:OK|ERR_[A-Z_]+)) \(?(-?\d+)\)?", src)}
    assert len(codes) == 8
    texts = {k: L.q3tts_strerror(v).decode() for k, v in codes.items()}
    assert texts["Q3TTS_OK"] == "ok"
    assert "unknown error" not in texts.values()
    assert len(set(texts.values())) == len(texts)
    for v in (-8, -99, 1, 1 << 30):
        assert L.q3tts_strerror(v).decode() == "unknown error"
