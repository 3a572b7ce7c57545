"""The frame-kernel trace summary (autoregressive_tts_decode_gb300.trace) on a
hand-built trace: step kinds decoded from the step marks, work = step start to
grid-barrier arrival, wait = arrival to the next step, ring waits attributed to
the step before their record."""
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
