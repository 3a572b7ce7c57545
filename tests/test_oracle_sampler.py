"""Pins of the oracle's sampler (CPU only).

The sampling controls are those of ``GenerateOptions`` in the "qwen3-tts-hip"
README, section "Library Usage" (do_sample, top_k, top_p, temperature,
repetition_penalty; the subtalker_* set for acoustic codes).  The checks below
tie the oracle's float rule to things fixed outside it: the softmax measure of
each token (exhaustive on V = 8), closed-form top-p and penalty examples, and
the limits in which sampling reduces to argmax.
"""
import math

import numpy as np
import pytest

pytestmark = pytest.mark.filterwarnings("ignore")


def _probs(logits, T):
    z = np.asarray(logits, dtype=np.float64) / T
    z = np.exp(z - z.max())
    return z / z.sum()


def test_expf_accuracy(oracle_mod):
    # Cody-Waite + degree-7 polynomial: within a few ulp of the true exp over [-80, 0].
    xs = np.concatenate([np.linspace(-80.0, 0.0, 20001, dtype=np.float32),
                         np.float32([0.0, -1e-8, -0.5, -1.0, -math.log(2), -10.25])])
    worst = 0.0
    for x in xs:
        got = oracle_mod.expf(float(x))
        ref = math.exp(float(x))
        ulp = np.spacing(np.float32(ref))
        worst = max(worst, abs(got - ref) / float(ulp))
    assert worst <= 2.0, worst
    assert oracle_mod.expf(0.0) == 1.0
    assert oracle_mod.expf(-100.0) == 0.0
    assert oracle_mod.expf(float("-inf")) == 0.0


def test_greedy_is_argmax_lowest_index(oracle_mod):
    lg = np.float32([0.1, 0.7, -0.3, 0.7, 0.2])
    assert oracle_mod.sample(lg, False, 50, 1.0, 0.9) == 1
    rng = np.random.default_rng(0)
    for _ in range(50):
        lg = rng.normal(size=3072).astype(np.float32)
        assert oracle_mod.sample(lg, False, 0, 1.0, 1.0) == int(np.argmax(lg))


def test_exhaustive_measure_v8(oracle_mod):
    """V = 8, no top-k/top-p: the set of u in [0,1) mapped to token i has measure
    p_i = softmax(l/T)_i, checked on a 2^-16 grid of u."""
    rng = np.random.default_rng(1)
    for trial in range(4):
        lg = rng.normal(scale=2.0, size=8).astype(np.float32)
        T = [1.0, 0.9, 0.5, 2.0][trial]
        p = _probs(lg, T)
        n = 1 << 16
        counts = np.zeros(8)
        picks = []
        for k in range(n):
            i = oracle_mod.sample(lg, True, 0, 1.0, T, u=k / n)
            counts[i] += 1
            picks.append(i)
        assert np.allclose(counts / n, p, atol=2.0 / n + 1e-6), (counts / n, p)
        # the map u -> token is monotone in the (value desc, index asc) order
        order = np.lexsort((np.arange(8), -(lg.astype(np.float64) / T)))
        rank = {int(t): r for r, t in enumerate(order)}
        ranks = [rank[i] for i in picks]
        assert all(a <= b for a, b in zip(ranks, ranks[1:]))


def test_top_k_one_is_argmax(oracle_mod):
    rng = np.random.default_rng(2)
    for _ in range(30):
        lg = rng.normal(size=2048).astype(np.float32)
        for u in (0.0, 0.3, 0.999999):
            assert oracle_mod.sample(lg, True, 1, 1.0, 0.9, u=u) == int(np.argmax(lg))


def test_top_p_tiny_is_argmax(oracle_mod):
    rng = np.random.default_rng(3)
    for _ in range(30):
        lg = rng.normal(size=2048).astype(np.float32)
        assert oracle_mod.sample(lg, True, 0, 1e-9, 0.9, u=0.99) == int(np.argmax(lg))


def test_top_p_closed_form(oracle_mod):
    # p = (0.5, 0.3, 0.2), top_p 0.6: the smallest prefix reaching 0.6 is {0, 1};
    # renormalised, u < 0.625 -> 0, else 1; token 2 is never drawn.
    lg = np.log(np.float64([0.5, 0.3, 0.2])).astype(np.float32)
    for u, want in ((0.0, 0), (0.6, 0), (0.62, 0), (0.63, 1), (0.9, 1), (0.9999, 1)):
        assert oracle_mod.sample(lg, True, 0, 0.6, 1.0, u=u) == want, u
    # top_p exactly 1.0 disables the filter: token 2 is reachable.
    assert oracle_mod.sample(lg, True, 0, 1.0, 1.0, u=0.9) == 2


def test_top_k_ties_keep_lowest_index(oracle_mod):
    lg = np.float32([1.0, 3.0, 3.0, 3.0, 0.0])
    # k = 2 keeps ids 1 and 2 (equal values, lower indices first) with equal weight.
    assert oracle_mod.sample(lg, True, 2, 1.0, 1.0, u=0.25) == 1
    assert oracle_mod.sample(lg, True, 2, 1.0, 1.0, u=0.75) == 2
    assert oracle_mod.sample(lg, True, 2, 1.0, 1.0, u=0.9999) == 2


def test_low_temperature_is_greedy(oracle_mod):
    rng = np.random.default_rng(4)
    for _ in range(30):
        lg = rng.normal(size=3072).astype(np.float32)
        for u in (0.0, 0.5, 0.999):
            assert oracle_mod.sample(lg, True, 50, 1.0, 1e-4, u=u) == int(np.argmax(lg))


def test_repetition_penalty_rule(oracle_mod):
    hist = np.zeros(4, dtype=np.uint8)
    hist[[0, 2]] = 1
    # positive logit divided: 1.0/1.05 < 0.99 -> id 1 wins over id 0
    lg = np.float32([1.0, 0.99, -5.0, -6.0])
    assert oracle_mod.sample(lg, False, 0, 1.0, 1.0, 1.05, hist) == 1
    assert oracle_mod.sample(lg, False, 0, 1.0, 1.0, 1.0, hist) == 0
    # negative logit multiplied: -1.0 * 1.05 < -1.02 -> id 3 wins over id 2
    lg = np.float32([-9.0, -9.0, -1.0, -1.02])
    assert oracle_mod.sample(lg, False, 0, 1.0, 1.0, 1.05, hist) == 3
    assert oracle_mod.sample(lg, False, 0, 1.0, 1.0, 1.0, hist) == 2
    # sampled: the penalised weight of id 0 is exp(1/1.05 - 1) relative to id 1 = exp(0)
    lg = np.float32([1.0, 1.0])
    h2 = np.uint8([1, 0])
    p0 = math.exp(1.0 / 1.05) / (math.exp(1.0 / 1.05) + math.exp(1.0))
    assert oracle_mod.sample(lg, True, 0, 1.0, 1.0, 1.05, h2, u=p0 - 1e-4) == 1  # id 1 ranks first
    assert oracle_mod.sample(lg, True, 0, 1.0, 1.0, 1.05, h2, u=(1 - p0) + 1e-4) == 0


def test_float_rule_matches_double_rule_away_from_boundaries(oracle_mod):
    rng = np.random.default_rng(5)
    n = 0
    for trial in range(300):
        V = 3072 if trial % 2 == 0 else 2048
        lg = rng.normal(scale=1.5, size=V).astype(np.float32)
        hist = (rng.random(V) < 0.05).astype(np.uint8)
        u = float(np.float32(rng.random()))
        a = oracle_mod.sample(lg, True, 50, 1.0, 0.9, 1.05, hist, u)
        b, margin = oracle_mod.sample_f64(lg, True, 50, 1.0, 0.9, 1.05, hist, u)
        if a != b:
            assert margin < 1e-5, (trial, margin)
        else:
            n += 1
    assert n >= 295


# --- special codes and the end-of-stream code (stop conditions) -------------
# Reading adopted: codes >= special_from are special; of them only eos_token may
# be drawn.  The candidate set is the allowed codes, so the draw is the same
# rule over the allowed codes alone.

def test_masked_measure_v8(oracle_mod):
    """V = 8, special_from = 5, eos_token = 6: the measure of u mapped to token
    i is softmax over the allowed codes {0..4, 6} (zero for 5 and 7), checked on
    a 2^-14 grid of u, with top-k disabled (0) and with k >= the allowed count."""
    rng = np.random.default_rng(11)
    allowed = np.array([1, 1, 1, 1, 1, 0, 1, 0], dtype=bool)
    for trial in range(3):
        lg = rng.normal(scale=2.0, size=8).astype(np.float32)
        lg[7] = lg.max() + 3.0  # a special code that would otherwise dominate
        T = [1.0, 0.7, 1.6][trial]
        z = np.where(allowed, lg.astype(np.float64) / T, -np.inf)
        p = np.exp(z - z.max())
        p /= p.sum()
        n = 1 << 14
        for k_top in (0, 6, 8):
            counts = np.zeros(8)
            for k in range(n):
                counts[oracle_mod.sample(lg, True, k_top, 1.0, T, u=k / n, special_from=5, eos_token=6)] += 1
            assert counts[5] == 0 and counts[7] == 0
            assert np.allclose(counts / n, p, atol=2.0 / n + 1e-6), (k_top, counts / n, p)
        # u just below 1 still picks an allowed code (the fallback is the last allowed kept)
        assert allowed[oracle_mod.sample(lg, True, 0, 1.0, T, u=1.0 - 2 ** -24, special_from=5, eos_token=6)]


def test_masked_greedy_and_eos_allowed(oracle_mod):
    lg = np.array([0.1, 0.5, 0.2, 3.0, 2.0, 1.0], dtype=np.float32)
    # codes 3.. are special: 3 and 5 are masked, 4 is the end-of-stream code
    assert oracle_mod.sample(lg, False, 0, 1.0, 1.0, special_from=3, eos_token=4) == 4
    assert oracle_mod.sample(lg, False, 0, 1.0, 1.0, special_from=3, eos_token=-1) == 1
    assert oracle_mod.sample(lg, False, 0, 1.0, 1.0) == 3  # no masking
    # top-k 1 over the allowed codes is their argmax
    assert oracle_mod.sample(lg, True, 1, 1.0, 1.0, u=0.99, special_from=3, eos_token=4) == 4


def test_end_of_stream_frames(oracle_mod):
    """A frame whose fed semantic code is eos_token yields [c0, -1 x 15] and ends
    the stream; later frames yield sixteen -1 and leave the stream's state as it
    was; a prefill restarts it."""
    import dataclasses
    from autoregressive_tts_decode_gb300 import synth
    shape = synth.WORKLOADS["tiny"].shape
    W = synth.make_weights(shape)
    p = synth.make_prompts(shape, [8])[0].numpy()
    u = synth.uniforms([0], 4)[0]
    eos = 777
    sp = dataclasses.replace(synth.GREEDY, eos_token=eos, special_from=0)
    orc = oracle_mod.Oracle(shape, W, 1, 64)
    orc.prefill(0, p)
    c0, _ = orc.step_frame(0, sp, u[0])
    assert (c0 >= 0).all()
    forced = c0.copy()
    forced[0] = eos
    h_before, l_before = orc.pending(0)
    n_before = orc.length(0)
    c1, _ = orc.step_frame(0, sp, u[1], forced=forced)
    assert (c1[1:] == -1).all() and c1[0] >= 0
    c2, _ = orc.step_frame(0, sp, u[2])
    assert (c2 == -1).all()
    h_after, l_after = orc.pending(0)
    assert orc.length(0) == n_before
    assert np.array_equal(h_before, h_after) and np.array_equal(l_before, l_after)
    # a prefill restarts the stream: the same first frame as before
    orc.prefill(0, p)
    c3, _ = orc.step_frame(0, sp, u[0])
    assert np.array_equal(c3, c0)
    # without an end-of-stream code the forced code is an ordinary semantic code
    orc2 = oracle_mod.Oracle(shape, W, 1, 64)
    orc2.prefill(0, p)
    orc2.step_frame(0, synth.GREEDY, u[0])
    c4, _ = orc2.step_frame(0, synth.GREEDY, u[1], forced=forced)
    assert (c4 >= 0).all()
