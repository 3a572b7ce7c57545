"""The frame-kernel trace summary (autoregressive_tts_decode_gb300.trace) on a
hand-built trace: step kinds decoded from the step marks, work = step start to
grid-barrier arrival, wait = arrival to the next step, ring waits attributed to
the step before their record; grid-barrier skew and release times from the
globaltimer."""
import numpy as np

from autoregressive_tts_decode_gb300 import trace as T


def _rec(tag, aux, clk):
    return [0, 0, clk, (tag << 16) | aux]


def test_step_table_on_a_hand_built_trace():
    mhz = 1000.0  # 1 cycle = 1 ns
    qkv, attn, ffn_t = 2 | (3 << 4), 3 | (3 << 4), 4 | (T.TALKER_PASS << 4)
    rows = [
        _rec(T.TR_STEP, T.FRAME_START, 0),
        _rec(T.TR_STEP, qkv, 1000),            # QKV: no barrier, ends at the next step
        _rec(T.TR_CW, 125, 3900),              # 125 x 16 cycles of ring wait in QKV
        _rec(T.TR_STEP, attn, 4000),           # CP_ATTN: arrives at 6000, next step at 9000
        _rec(T.TR_ARRIVE, 0, 6000),
        _rec(4, 0, 8500),                      # (the barrier's pass mark is not needed)
        _rec(T.TR_STEP, ffn_t, 9000),          # the Talker's FFN
        _rec(T.TR_ARRIVE, 0, 12000),
        _rec(T.TR_STEP, 1 | (3 << 4), 14000),  # a last step closes the FFN
    ]
    tr = np.zeros((2, T.TRACE_EV, 4), dtype=np.uint32)
    tr[0, :len(rows)] = np.array(rows, dtype=np.uint32)
    tab = T.step_table(tr, mhz=mhz)
    assert set(tab) == {"QKV", "CP_ATTN", "FFN_T"}
    n, work, wait, ring = tab["QKV"]
    assert (n, work, wait, ring) == (1.0, 3.0, 0.0, 2.0)
    assert tab["CP_ATTN"][1:3] == (2.0, 3.0)
    assert tab["FFN_T"][1:3] == (3.0, 2.0)


def test_step_kinds_follow_the_kernel_enum():
    assert T.step_kind(0) == "DRAW" and T.step_kind(0 | (T.TALKER_PASS << 4)) == "DRAW_T"
    assert T.step_kind(8) == "T_HEAD" and T.step_kind(6 | (T.TALKER_PASS << 4)) == "T_ATTN"


def _grec(tag, aux, ns):
    return [ns & 0xFFFFFFFF, ns >> 32, 0, (tag << 16) | aux]


def test_barrier_table_on_a_hand_built_trace():
    """Skew, spread and release of grid barriers from globaltimer records of
    three CTAs, with the timer's epoch-sized base (about 1.8e18 ns), which
    float64 cannot hold to the nanosecond."""
    base = 1_780_000_000_000_000_000
    attn, ffn = 3 | (2 << 4), 4 | (2 << 4)
    times = [  # per CTA: (arrive, pass) of the attention barrier, then of the FFN barrier
        ((1000, 3000), (5000, 8000)),
        ((1200, 3100), (5600, 8000)),
        ((2000, 3050), (5200, 8100)),
    ]
    tr = np.zeros((4, T.TRACE_EV, 4), dtype=np.uint32)
    for c, ((a0, p0), (a1, p1)) in enumerate(times):
        rows = [_grec(T.TR_STEP, T.FRAME_START, base), _grec(T.TR_STEP, attn, base + 500),
                _grec(T.TR_ARRIVE, 0, base + a0), _grec(T.TR_PASS, 0, base + p0),
                _grec(T.TR_STEP, ffn, base + p0 + 10),
                _grec(T.TR_ARRIVE, 0, base + a1), _grec(T.TR_PASS, 0, base + p1)]
        tr[c, :len(rows)] = np.array(rows, dtype=np.uint64).astype(np.uint32)
    tab = T.barrier_table(tr)
    assert list(tab) == ["CP_ATTN", "FFN"]
    # arrivals 1000/1200/2000 ns: skew 2000 - 1200, spread 1000, release 3000 - 2000
    assert tab["CP_ATTN"] == (1.0, 0.8, 1.0, 1.0)
    # arrivals 5000/5600/5200 ns: skew 5600 - 5200, spread 600, release 8000 - 5600
    assert tab["FFN"] == (1.0, 0.4, 0.6, 2.4)


def test_interval_table_adds_up_to_the_frame():
    """Two CTAs, two barriers and an end mark: the intervals (slowest CTA's work
    + release) and the tail add up to the frame, first start to last end."""
    base = 1_780_000_000_000_000_000
    qkv, attn, ffn, head = 2 | (3 << 4), 3 | (3 << 4), 4 | (3 << 4), 5 | (3 << 4)
    ctas = [
        [(T.TR_STEP, T.FRAME_START, 0), (T.TR_STEP, qkv, 10), (T.TR_STEP, attn, 100),
         (T.TR_ARRIVE, 0, 300), (T.TR_PASS, 0, 500), (T.TR_STEP, ffn, 510),
         (T.TR_ARRIVE, 0, 900), (T.TR_PASS, 0, 1200), (T.TR_STEP, head, 1210), (T.TR_END, 0, 1400)],
        [(T.TR_STEP, T.FRAME_START, 5), (T.TR_STEP, qkv, 12), (T.TR_STEP, attn, 110),
         (T.TR_ARRIVE, 0, 400), (T.TR_PASS, 0, 520), (T.TR_STEP, ffn, 530),
         (T.TR_ARRIVE, 0, 1000), (T.TR_PASS, 0, 1210), (T.TR_STEP, head, 1220), (T.TR_END, 0, 1500)],
    ]
    tr = np.zeros((3, T.TRACE_EV, 4), dtype=np.uint32)
    for c, recs in enumerate(ctas):
        tr[c, :len(recs)] = np.array([_grec(t, a, base + ns) for t, a, ns in recs],
                                     dtype=np.uint64).astype(np.uint32)
    tab, tail = T.interval_table(tr)
    assert tab == {"QKV+CP_ATTN": (1, 0.4, 0.1), "FFN": (1, 0.5, 0.2)}
    assert tail == 0.3
    assert sum(w + r for _, w, r in tab.values()) + tail == 1.5  # first start 0 to last end 1500 ns
