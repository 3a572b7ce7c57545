"""Pins of the oracle's model arithmetic (CPU only).

Each check ties the oracle to something outside itself: library routines
(torch's rms_norm, scaled_dot_product_attention, silu, linear) on cases the
layer reduces to, closed forms of the rotation, invariants, and whole-model
special cases where zeroed weights reduce a frame to plain lookups and matrix
products.  Frame structure: "Running Qwen3-TTS on an AMD R9700", section
"Running Qwen3-TTS" (16 codes per frame, Talker then 15 CodePredictor steps);
embedding sum: "qwen3-tts-hip" README, section "Python Parity Fixtures".
"""
import dataclasses
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from autoregressive_tts_decode_gb300 import synth

TINY = synth.WORKLOADS["tiny"]


def f64(t):
    return t.detach().to(torch.float64).numpy()


def test_rmsnorm_matches_library_and_invariants(oracle_mod):
    rng = np.random.default_rng(0)
    x = rng.normal(size=256) * 3.0
    g = rng.normal(size=256).astype(np.float32)
    y = oracle_mod.rmsnorm(x, g, 1e-6)
    ref = F.rms_norm(torch.tensor(x), (256,), torch.tensor(g, dtype=torch.float64), eps=1e-6)
    assert np.allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)
    y1 = oracle_mod.rmsnorm(x, np.ones(256, np.float32), 1e-6)
    assert abs(math.sqrt(np.mean(y1 ** 2)) - 1.0) < 1e-6
    y2 = oracle_mod.rmsnorm(x * 37.5, np.ones(256, np.float32), 1e-6)
    assert np.allclose(y1, y2, rtol=1e-6)


def test_rope_closed_form_and_invariants(oracle_mod):
    theta = 1e6
    # hd = 4: pairs (0, 2) at frequency 1 and (1, 3) at theta^-1/2.
    for pos in (0, 1, 7, 300):
        e0 = oracle_mod.rope(np.array([1.0, 0, 0, 0]), pos, theta)
        assert np.allclose(e0, [math.cos(pos), 0, math.sin(pos), 0], atol=1e-12)
        e1 = oracle_mod.rope(np.array([0, 1.0, 0, 0]), pos, theta)
        a = pos * theta ** -0.5
        assert np.allclose(e1, [0, math.cos(a), 0, math.sin(a)], atol=1e-12)
        e2 = oracle_mod.rope(np.array([0, 0, 1.0, 0]), pos, theta)
        assert np.allclose(e2, [-math.sin(pos), 0, math.cos(pos), 0], atol=1e-12)
    rng = np.random.default_rng(1)
    q = rng.normal(size=128)
    k = rng.normal(size=128)
    assert np.allclose(oracle_mod.rope(q, 0, theta), q)
    for pos in (1, 100, 2047):
        r = oracle_mod.rope(q, pos, theta)
        assert abs(np.linalg.norm(r) - np.linalg.norm(q)) < 1e-10
    # q(m) . k(n) depends on m - n only
    d1 = oracle_mod.rope(q, 50, theta) @ oracle_mod.rope(k, 45, theta)
    d2 = oracle_mod.rope(q, 1005, theta) @ oracle_mod.rope(k, 1000, theta)
    assert abs(d1 - d2) < 1e-9


@pytest.mark.parametrize("Hq,Hkv,S", [(4, 2, 1), (4, 2, 37), (16, 8, 200), (8, 8, 9)])
def test_attention_matches_sdpa(oracle_mod, Hq, Hkv, S):
    rng = np.random.default_rng(S)
    hd = 64
    q = rng.normal(size=(Hq, hd))
    K = rng.normal(size=(S, Hkv, hd))
    V = rng.normal(size=(S, Hkv, hd))
    o = oracle_mod.attention(q, K, V)
    qt = torch.tensor(q)[None, :, None, :]
    kt = torch.tensor(K).permute(1, 0, 2)[None]
    vt = torch.tensor(V).permute(1, 0, 2)[None]
    ref = F.scaled_dot_product_attention(qt, kt, vt, enable_gqa=(Hq != Hkv))[0, :, 0, :]
    assert np.allclose(o, ref.numpy(), rtol=1e-10, atol=1e-10)
    if S == 1:
        # softmax over a single position: the output is that position's v
        assert np.allclose(o, np.repeat(V[0], Hq // Hkv, axis=0), atol=1e-12)


def _tiny_weights(dtype=synth.DTYPE_F32, **zero):
    W = synth.make_weights(dataclasses.replace(TINY.shape, weight_dtype=dtype))
    for name in list(W):
        for key, layers in zero.items():
            if name.endswith("." + key) and name.split(".")[0] in layers:
                W[name] = torch.zeros_like(W[name])
    return W


def mat(W, name, j=None):
    """A weight matrix as torch float64 through torch's own conversions: FP8
    codes (uint8 storage) through float8_e4m3fn -> float64 times the row scales
    (synth.SCALE_OF); bf16 / fp32 directly.  j picks one head of a stacked
    tensor."""
    t = W[name] if j is None else W[name][j]
    if t.dtype == torch.uint8:
        sname = name.rsplit(".", 1)[0] + "." + synth.SCALE_OF[name.rsplit(".", 1)[1]]
        sc = W[sname] if j is None else W[sname][j]
        return t.view(torch.float8_e4m3fn).to(torch.float64) * sc.to(torch.float64).unsqueeze(-1)
    return t.to(torch.float64)


def _rms(x, g, eps=1e-6):
    return F.rms_norm(torch.tensor(x, dtype=torch.float64), (x.shape[-1],),
                      torch.tensor(g, dtype=torch.float64), eps=eps).numpy()


def test_identity_stack_gives_head_of_normed_input(oracle_mod):
    """With W_o = W_down = 0 every Talker layer is the identity, so the pending
    logits are W_head . RMSNorm(last prompt vector) * g_final."""
    s = TINY.shape
    W = _tiny_weights(w_o=("talker",), w_down=("talker",))
    o = oracle_mod.Oracle(s, W, 1, TINY.kv_cap)
    p = synth.make_prompts(s, [5])[0].numpy()
    o.prefill(0, p)
    h, lg = o.pending(0)
    hn = _rms(p[-1].astype(np.float64), f64(W["talker.g_final"]))
    assert np.allclose(h, hn, rtol=1e-10, atol=1e-12)
    assert np.allclose(lg, f64(W["talker.w_head"]) @ hn, rtol=1e-9, atol=1e-12)


@pytest.mark.parametrize("dtype", [synth.DTYPE_F32, synth.DTYPE_BF16, synth.DTYPE_FP8])
def test_single_position_attention_block(oracle_mod, dtype):
    """Prompt of length 1 and W_down = 0: attention over one position returns v,
    so x = e + W_o v with v = W_v RMSNorm(e) (the v rows of W_qkv).  With bf16
    weights the expected value widens them through torch, not the oracle."""
    s = dataclasses.replace(TINY.shape, talker_layers=1, weight_dtype=dtype)
    W = _tiny_weights(dtype, w_down=("talker",))
    W = {k: v for k, v in W.items() if not k.startswith("talker.1.")}
    o = oracle_mod.Oracle(s, W, 1, TINY.kv_cap)
    e = synth.make_prompts(s, [1])[0].numpy().astype(np.float64)
    x = o.talker_stack(0, e, 0)[0]
    n = _rms(e[0], f64(W["talker.0.g_attn_norm"]))
    vrows = mat(W, "talker.0.w_qkv").numpy()[(s.n_q_heads + s.n_kv_heads) * s.head_dim:]
    v = (vrows @ n).reshape(s.n_kv_heads, s.head_dim)
    o_heads = np.repeat(v, s.n_q_heads // s.n_kv_heads, axis=0).reshape(-1)
    want = e[0] + mat(W, "talker.0.w_o").numpy() @ o_heads
    assert np.allclose(x, want, rtol=1e-9, atol=1e-12)


@pytest.mark.parametrize("dtype", [synth.DTYPE_F32, synth.DTYPE_BF16, synth.DTYPE_FP8])
def test_ffn_block_is_swiglu(oracle_mod, dtype):
    """W_o = 0 leaves the FFN: x = e + W_down(silu(W_gate n) * W_up n), n = RMSNorm(e)."""
    s = dataclasses.replace(TINY.shape, talker_layers=1, weight_dtype=dtype)
    W = _tiny_weights(dtype, w_o=("talker",))
    W = {k: v for k, v in W.items() if not k.startswith("talker.1.")}
    o = oracle_mod.Oracle(s, W, 1, TINY.kv_cap)
    e = synth.make_prompts(s, [3])[0].to(torch.float64)
    x = o.talker_stack(0, e.numpy(), 0)
    n = F.rms_norm(e, (s.talker_hidden,), W["talker.0.g_ffn_norm"].double(), eps=1e-6)
    gu = F.linear(n, mat(W, "talker.0.w_gateup"))
    a = F.silu(gu[:, :s.talker_ffn]) * gu[:, s.talker_ffn:]
    want = e + F.linear(a, mat(W, "talker.0.w_down"))
    assert np.allclose(x, want.numpy(), rtol=1e-9, atol=1e-12)


def _embed_sum(W, codes):
    x = f64(W["talker.e_codec"])[codes[0]].copy()
    for j in range(1, 16):
        x += f64(W["cp.embeds"][j - 1])[codes[j]]
    return x


@pytest.mark.parametrize("dtype", [synth.DTYPE_F32, synth.DTYPE_BF16, synth.DTYPE_FP8])
@pytest.mark.parametrize("proj", [False, True])
def test_frame_wiring_with_identity_stacks(oracle_mod, proj, dtype):
    """Both stacks reduced to the identity (W_o = W_down = 0): each CodePredictor
    logit vector is head_j . RMSNorm(P u_j) with u_0 = E_t[c0] (pass 0's last token)
    and u_j = E_cp[j-1][c_j]; the next pending logits are the codec head of the
    normed embedding sum of the frame's 16 codes.  For bf16 storage the
    expected values come from torch's own bf16 -> fp64 conversion of the same
    tensors, so a wrong shift or half-word order in the oracle's widening of
    bf16 weights fails here."""
    shape = dataclasses.replace(TINY.shape, weight_dtype=dtype)
    if proj:
        shape = dataclasses.replace(shape, cp_hidden=128, cp_ffn=384)
    W = synth.make_weights(shape)
    for name in list(W):
        if name.endswith(".w_o") or name.endswith(".w_down"):
            W[name] = torch.zeros_like(W[name])
    o = oracle_mod.Oracle(shape, W, 1, TINY.kv_cap)
    o.prefill(0, synth.make_prompts(shape, [4])[0].numpy())
    _, l0 = o.pending(0)
    u = synth.uniforms([0], 1)[0, 0]
    codes, lg = o.step_frame(0, synth.GREEDY, u, want_logits=True)
    assert codes.shape == (16,)
    assert np.array_equal(lg[:shape.codec_vocab], l0.astype(np.float32))
    assert codes[0] == int(np.argmax(l0.astype(np.float32)))
    Vt, Vc = shape.codec_vocab, shape.cp_vocab
    for j in range(15):
        u_j = (f64(W["talker.e_codec"])[codes[0]] if j == 0
               else f64(W["cp.embeds"][j - 1])[codes[j]])
        z = mat(W, "cp.w_proj").numpy() @ u_j if proj else u_j
        want = mat(W, "cp.heads", j).numpy() @ _rms(z, f64(W["cp.g_final"]))
        got = lg[Vt + j * Vc: Vt + (j + 1) * Vc]
        assert np.allclose(got, want, rtol=1e-5, atol=1e-6), j
        assert codes[j + 1] == int(np.argmax(got))
    _, l1 = o.pending(0)
    x = _embed_sum(W, codes)
    want = mat(W, "talker.w_head").numpy() @ _rms(x, f64(W["talker.g_final"]))
    assert np.allclose(l1, want, rtol=1e-9, atol=1e-12)


def test_incremental_talker_equals_full_recompute(oracle_mod):
    """prefill(n) + k teacher-forced frames leaves the same pending state as one
    prefill of the n prompt vectors followed by the k embedding sums."""
    s = TINY.shape
    W = synth.make_weights(s)
    prompt = synth.make_prompts(s, [9])[0].numpy()
    rng = np.random.default_rng(7)
    forced = [np.concatenate([[rng.integers(0, s.codec_vocab)], rng.integers(0, s.cp_vocab, 15)])
              .astype(np.int32) for _ in range(4)]
    a = oracle_mod.Oracle(s, W, 1, TINY.kv_cap)
    a.prefill(0, prompt)
    u = synth.uniforms([0], 4)[0]
    for f in range(4):
        a.step_frame(0, synth.GREEDY, u[f], forced=forced[f])
    ha, la = a.pending(0)
    seq = np.concatenate([prompt.astype(np.float64)] + [_embed_sum(W, c)[None] for c in forced])
    b = oracle_mod.Oracle(s, W, 1, TINY.kv_cap)
    b.prefill(0, seq.astype(np.float32))
    hb, lb = b.pending(0)
    # the float32 cast of the embedding sums is the only difference
    assert np.allclose(la, lb, atol=2e-5)
    assert np.allclose(ha, hb, atol=2e-5)
    assert a.length(0) == b.length(0) == 13


def test_incremental_codepredictor_equals_full_pass(oracle_mod):
    """The 15 cached CodePredictor passes of a frame give the same logits as one
    causal pass over [h_T, E_t[c0], E_cp[0][c1], ..., E_cp[13][c14]]."""
    for shape in (TINY.shape, dataclasses.replace(TINY.shape, cp_hidden=128, cp_ffn=384)):
        W = synth.make_weights(shape)
        o = oracle_mod.Oracle(shape, W, 1, TINY.kv_cap)
        o.prefill(0, synth.make_prompts(shape, [6])[0].numpy())
        h, _ = o.pending(0)
        codes, lg = o.step_frame(0, synth.GREEDY, synth.uniforms([0], 1)[0, 0], want_logits=True)
        toks = [h, f64(W["talker.e_codec"])[codes[0]]]
        toks += [f64(W["cp.embeds"][j - 1])[codes[j]] for j in range(1, 15)]
        full = o.cp_full(np.stack(toks))
        inc = lg[shape.codec_vocab:].reshape(15, shape.cp_vocab)
        assert np.allclose(inc, full, atol=1e-6)


def test_frame_determinism_and_shape(oracle_mod):
    s = TINY.shape
    W = synth.make_weights(s)
    runs = []
    for _ in range(2):
        o = oracle_mod.Oracle(s, W, 1, TINY.kv_cap)
        o.prefill(0, synth.make_prompts(s, [16])[0].numpy())
        u = synth.uniforms([0], 3)[0]
        runs.append(np.stack([o.step_frame(0, synth.QWEN_DEFAULT_SAMPLING, u[f])[0]
                              for f in range(3)]))
    assert np.array_equal(runs[0], runs[1])
    assert runs[0].shape == (3, 16)
    assert runs[0][:, 0].max() < s.codec_vocab and runs[0][:, 1:].max() < s.cp_vocab


def test_capacity(oracle_mod):
    s = TINY.shape
    W = synth.make_weights(s)
    o = oracle_mod.Oracle(s, W, 1, 20)
    with pytest.raises(ValueError):
        o.prefill(0, np.zeros((20, s.talker_hidden), np.float32))
    o.prefill(0, synth.make_prompts(s, [18])[0].numpy())
    u = synth.uniforms([0], 3)[0]
    o.step_frame(0, synth.GREEDY, u[0])
    o.step_frame(0, synth.GREEDY, u[1])
    with pytest.raises(ValueError):
        o.step_frame(0, synth.GREEDY, u[2])


def _rotate_half(x, pos, theta):
    """Closed-form RoPE rotation of [..., hd] rows at the given positions."""
    hd = x.shape[-1]
    half = hd // 2
    inv = theta ** (-2.0 * np.arange(half) / hd)
    ang = np.asarray(pos, dtype=np.float64)[:, None] * inv[None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c[:, None, :] - b * s[:, None, :],
                           b * c[:, None, :] + a * s[:, None, :]], axis=-1)


@pytest.mark.parametrize("kv_bf16", [False, True])
def test_attention_block_with_qk_norm_and_causal_mask(oracle_mod, kv_bf16):
    """One Talker layer with W_down = 0 and non-unit q/k norm gains over a
    3-token prompt, rebuilt from library calls: rms_norm -> per-head rms_norm *
    gain -> rotation -> causal scaled_dot_product_attention -> W_o.  With a bf16
    cache (the serving configuration) the cached k, v enter the attention as
    torch's own fp32 -> bf16 round-to-nearest-even conversion of them."""
    s = dataclasses.replace(TINY.shape, talker_layers=1)
    W = _tiny_weights(w_down=("talker",))
    W = {k: v for k, v in W.items() if not k.startswith("talker.1.")}
    gen = torch.Generator().manual_seed(99)
    W["talker.0.g_q_norm"] = 1.0 + 0.5 * torch.randn(s.head_dim, generator=gen)
    W["talker.0.g_k_norm"] = 1.0 + 0.5 * torch.randn(s.head_dim, generator=gen)
    o = oracle_mod.Oracle(s, W, 1, TINY.kv_cap, kv_bf16=kv_bf16)
    T, Hq, Hkv, hd = 3, s.n_q_heads, s.n_kv_heads, s.head_dim
    e = synth.make_prompts(s, [T])[0].to(torch.float64)
    x = o.talker_stack(0, e.numpy(), 0)
    n = F.rms_norm(e, (s.talker_hidden,), W["talker.0.g_attn_norm"].double(), eps=1e-6)
    qkv = F.linear(n, W["talker.0.w_qkv"].double())
    q = qkv[:, :Hq * hd].reshape(T, Hq, hd)
    k = qkv[:, Hq * hd:(Hq + Hkv) * hd].reshape(T, Hkv, hd)
    v = qkv[:, (Hq + Hkv) * hd:].reshape(T, Hkv, hd)
    q = F.rms_norm(q, (hd,), W["talker.0.g_q_norm"].double(), eps=1e-6)
    k = F.rms_norm(k, (hd,), W["talker.0.g_k_norm"].double(), eps=1e-6)
    q = torch.tensor(_rotate_half(q.numpy(), np.arange(T), s.rope_theta))
    k = torch.tensor(_rotate_half(k.numpy(), np.arange(T), s.rope_theta))
    if kv_bf16:
        k = k.float().to(torch.bfloat16).double()
        v = v.float().to(torch.bfloat16).double()
    att = F.scaled_dot_product_attention(q.permute(1, 0, 2)[None], k.permute(1, 0, 2)[None],
                                         v.permute(1, 0, 2)[None], is_causal=True,
                                         enable_gqa=True)[0].permute(1, 0, 2).reshape(T, Hq * hd)
    want = e + F.linear(att, W["talker.0.w_o"].double())
    assert np.allclose(x, want.numpy(), rtol=1e-9, atol=1e-11)


def _penalty_case():
    """Identity stacks (W_o = W_down = 0 everywhere) and a hand-made codec head
    whose rows A and B carry a near tie: rows = s * u1 and 0.98 s * u1 + 3 s * u2
    for two orthonormal directions.  u1 is the direction of the embedding sum
    of a fixed forced frame (semantic code A, first acoustic code B), so after
    that frame the pending logits are l_A > l_B > 0 with l_B / l_A = 0.98; a
    prompt ending in u2 gives the pending logits l_B = 3 s |h| and l_A = 0, so
    the first frame draws B greedily.  All other rows are 0."""
    shape = TINY.shape
    W = synth.make_weights(shape)
    for name in list(W):
        if name.endswith(".w_o") or name.endswith(".w_down"):
            W[name] = torch.zeros_like(W[name])
    D, Vt = shape.talker_hidden, shape.codec_vocab
    A, B = 1234, 77
    rng = np.random.default_rng(5)
    forced = np.concatenate([[A, B], rng.integers(0, shape.cp_vocab, 14)]).astype(np.int32)
    x1 = _embed_sum(W, forced)
    u1 = x1 / np.linalg.norm(x1)
    r = rng.normal(size=D)
    u2 = r - (r @ u1) * u1
    u2 /= np.linalg.norm(u2)
    head = np.zeros((Vt, D))
    s = 0.05
    head[A] = s * u1
    head[B] = 0.98 * s * u1 + 3.0 * s * u2
    W["talker.w_head"] = torch.tensor(head, dtype=torch.float32)
    return shape, W, A, B, forced, u1, u2


def test_repetition_penalty_history_is_the_fed_semantic_code(oracle_mod):
    """Repetition penalty bookkeeping ("qwen3-tts-hip" README, "Library Usage",
    GenerateOptions::repetition_penalty; the usual divide-positive rule):
      * the history holds the semantic code fed forward (the forced one under
        teacher forcing), not the drawn one -- frame 1 draws B but feeds A;
      * it changes the next frame's pick: with rho = 1.5 the near tie A > B of
        frame 2 flips to B, with rho = 1 it stays A;
      * acoustic codes never enter it -- frame 1 feeds B as its first acoustic
        code, and a penalised B would turn the flip back to A;
      * prefill restarts it, and another stream's history is its own."""
    shape, W, A, B, forced, u1, u2 = _penalty_case()
    pen = dataclasses.replace(synth.GREEDY, repetition_penalty=1.5)
    u = synth.uniforms([0], 2)[0]
    prompt = np.zeros((3, shape.talker_hidden), np.float32)
    prompt[-1] = u2
    for rho, want2 in ((1.0, A), (1.5, B)):
        sp = dataclasses.replace(synth.GREEDY, repetition_penalty=rho)
        o = oracle_mod.Oracle(shape, W, 1, TINY.kv_cap)
        o.prefill(0, prompt)
        c1, _ = o.step_frame(0, sp, u[0], forced=forced)
        assert c1[0] == B  # drawn B, fed A
        _, l2 = o.pending(0)
        assert l2[A] > l2[B] > l2[A] / 1.5 > 0
        c2, _ = o.step_frame(0, sp, u[1])
        assert c2[0] == want2, (rho, c2[0])
    # a prompt ending in u1 gives the near tie A > B at once
    tie_prompt = np.zeros((2, shape.talker_hidden), np.float32)
    tie_prompt[-1] = u1
    o = oracle_mod.Oracle(shape, W, 2, TINY.kv_cap)
    o.prefill(0, prompt)
    o.step_frame(0, pen, u[0], forced=forced)  # history of stream 0: {A}
    o.prefill(1, tie_prompt)                    # stream 1 never fed A
    c, _ = o.step_frame(1, pen, u[0])
    assert c[0] == A
    o.prefill(0, tie_prompt)                    # stream 0 restarts: history cleared
    c, _ = o.step_frame(0, pen, u[0])
    assert c[0] == A


def test_fp8_decoder_all_codes(oracle_mod):
    """The oracle's E4M3 decoder on all 256 codes equals torch's float8_e4m3fn
    conversion (NaN exactly at 0x7f and 0xff; 448 the largest value)."""
    codes = torch.arange(256, dtype=torch.uint8)
    want = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle_mod.fp8_value(c) for c in range(256)])
    nan = np.isnan(want)
    assert list(np.nonzero(nan)[0]) == [0x7f, 0xff]
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert got[0x7e] == 448.0 and got[0x01] == 2.0 ** -9
