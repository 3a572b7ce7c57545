"""Shared helpers of the GPU parity tests: run the CUDA engine and the oracle on
the same seeded inputs and compare them."""
from __future__ import annotations

import numpy as np

from autoregressive_tts_decode_gb300 import synth


def gpu_weights(shape, seed=synth.SEED_WEIGHTS, gen_device="cpu"):
    """(cpu_weights, cuda_weights) with identical bytes."""
    import torch
    W = synth.make_weights(shape, seed=seed, device=gen_device)
    if gen_device == "cpu":
        return W, {k: v.to("cuda") for k, v in W.items()}
    return {k: v.cpu() for k, v in W.items()}, W


def run_gpu(eng, stream_ids, prompts, sampling, frames, forced=None, uniforms=None,
            prefill=True):
    """Prefills each stream, runs `frames` frames for all streams together.
    Returns codes [n, frames, 16] and logits [n, frames, V_t + 15 V_c] (numpy)."""
    import torch
    s = eng.shape
    n = len(stream_ids)
    if prefill:
        for sid, p in zip(stream_ids, prompts):
            eng.prefill(sid, p.to("cuda"))
    if uniforms is None:
        uniforms = synth.uniforms(stream_ids, frames)
    width = s.codec_vocab + 15 * s.cp_vocab
    codes = np.zeros((n, frames, 16), dtype=np.int32)
    logits = np.zeros((n, frames, width), dtype=np.float32)
    c = torch.zeros((n, 16), dtype=torch.int32, device="cuda")
    lg = torch.zeros((n, width), dtype=torch.float32, device="cuda")
    for f in range(frames):
        u = torch.from_numpy(np.ascontiguousarray(uniforms[:, f])).to("cuda")
        fc = None
        if forced is not None:
            fc = torch.from_numpy(np.ascontiguousarray(forced[:, f])).to("cuda")
        eng.step_frame(stream_ids, sampling, u, c, forced=fc, logits=lg)
        codes[:, f] = c.cpu().numpy()
        logits[:, f] = lg.cpu().numpy()
    eng.sync()
    return codes, logits


def run_oracle(orc, sid, prompt, sampling, frames, forced=None, uniforms=None):
    """Oracle run of one stream; returns codes [frames, 16], logits [frames, width]."""
    orc.prefill(sid, np.asarray(prompt, dtype=np.float32))
    if uniforms is None:
        uniforms = synth.uniforms([sid], frames)[0]
    codes, logits = [], []
    for f in range(frames):
        c, lg = orc.step_frame(sid, sampling, uniforms[f],
                               forced=None if forced is None else forced[f], want_logits=True)
        codes.append(c)
        logits.append(lg)
    return np.stack(codes), np.stack(logits)


def fed_codes(codes, forced):
    return codes if forced is None else forced


def sampler_replay(oracle_mod, shape, sampling, codes, logits, fed, uniforms):
    """Returns the number of draws where the oracle's rule on the GPU's own logits
    disagrees with the GPU's code (must be 0)."""
    Vt, Vc = shape.codec_vocab, shape.cp_vocab
    hist = np.zeros(Vt, dtype=np.uint8)
    bad = 0
    sf, eos = getattr(sampling, "special_from", 0), getattr(sampling, "eos_token", -1)
    for f in range(codes.shape[0]):
        lg = logits[f]
        c0 = oracle_mod.sample(lg[:Vt], sampling.do_sample, sampling.top_k, sampling.top_p,
                               sampling.temperature, sampling.repetition_penalty, hist,
                               float(uniforms[f, 0]), special_from=sf, eos_token=eos)
        bad += int(c0 != codes[f, 0])
        hist[fed[f, 0]] = 1
        for j in range(15):
            cj = oracle_mod.sample(lg[Vt + j * Vc: Vt + (j + 1) * Vc], sampling.sub_do_sample,
                                   sampling.sub_top_k, sampling.sub_top_p,
                                   sampling.sub_temperature, 1.0, None, float(uniforms[f, j + 1]))
            bad += int(cj != codes[f, j + 1])
    return bad


def logits_report(gpu_logits, ora_logits, shape, tie=3e-2):
    """(max abs error, argmax agreement over all 16 draws per frame).  A draw
    whose two argmaxes differ counts as agreeing when the oracle's logits at
    them are within 2 * tie of each other: each logit may be off by the
    tolerance, so a gap that small does not fix the argmax (a near-tie, where
    float reassociation from run to run may pick either)."""
    Vt, Vc = shape.codec_vocab, shape.cp_vocab
    err = float(np.max(np.abs(gpu_logits - ora_logits)))
    agree, total = 0, 0
    for f in range(gpu_logits.shape[0]):
        segs = [(0, Vt)] + [(Vt + j * Vc, Vt + (j + 1) * Vc) for j in range(15)]
        for a, b in segs:
            g, o = int(np.argmax(gpu_logits[f, a:b])), int(np.argmax(ora_logits[f, a:b]))
            near_tie = abs(float(ora_logits[f, a + g]) - float(ora_logits[f, a + o])) <= 2 * tie
            agree += int(g == o or near_tie)
            total += 1
    return err, agree / total
