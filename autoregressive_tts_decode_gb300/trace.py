"""Per-phase timeline of the persistent frame kernel, from a profiling build.

Built with -DQ3TTS_TRACE, the kernel has consumer thread 0 of every CTA append
a record {globaltimer low, globaltimer high, clock64 low, tag << 16 | aux} at
phase boundaries for the last frame launched (FK_MARK in csrc/frame_kernel.cu):
the start of each step (aux = step kind | pass << 4 | layer << 9; aux 15 the
frame start), the arrival at and the passing of each grid barrier, marks inside
steps, and, before each step, the longest time one consumer warp of the CTA
spent waiting for ring data in the step before (aux in units of 16 clock64
cycles).  This module builds that library beside the normal one (under
_build/trace/), runs frames of a workload on it, and tabulates per step kind
the median time from a step's start to its grid-barrier arrival (work) and
from there to the next step's start (wait), and per grid barrier the CTAs'
arrival skew and the release time from the last arrival to the first pass
(globaltimer, one clock for all SMs), and the frame split into the intervals
between barriers, which add up to the whole frame.  Each mark costs about 0.1 us, so a
traced frame runs slower than a plain one.

    python -m autoregressive_tts_decode_gb300.trace --workload 1.7b --frames 12
"""
from __future__ import annotations

import argparse
import collections
import ctypes as C
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Tuple

import numpy as np

from . import build

# the kernel's trace buffer: FK_MAXCTA rows of FK_TRACE_EV records of 4 words
MAXCTA, TRACE_EV = 256, 8192
# record tags (TR_* in csrc/frame_kernel.cu)
TR_STEP, TR_ARRIVE, TR_PASS, TR_END, TR_CW = 1, 3, 4, 7, 8
FRAME_START = 15  # the aux of the frame's opening TR_STEP
# step kinds in the kernel's order (enum StepKind); the Talker's draw, QKV and
# FFN steps (pass 15) get a "_T" suffix
KINDS = ["DRAW", "PROJ", "QKV", "CP_ATTN", "FFN", "CP_HEAD", "T_ATTN", "T_OPROJ", "T_HEAD"]
TALKER_PASS = 15


def build_traced() -> str:
    """Compiles the library with -DQ3TTS_TRACE into _build/trace/; returns its path."""
    out = os.path.join(build.BUILD, "trace")
    os.makedirs(out, exist_ok=True)
    lib = os.path.join(out, "libq3tts_trace.so")
    srcs = build.sources()
    objs = [os.path.join(out, os.path.basename(s)[:-3] + ".o") for s in srcs]

    def compile_one(pair):
        src, obj = pair
        return subprocess.run([build.NVCC, *build.ARCH, *build.FLAGS, "-DQ3TTS_TRACE", "-c", src, "-o", obj],
                              capture_output=True, text=True)

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, zip(srcs, objs)))
    bad = [r.stderr for r in results if r.returncode != 0]
    if bad:
        raise RuntimeError("nvcc failed:\n" + "\n".join(bad))
    subprocess.run([build.NVCC, *build.ARCH, "-shared", "-o", lib, *objs], check=True)
    return lib


def capture(workload: str = "1.7b", frames: int = 12):
    """Runs `frames` frames of one stream of the workload on the traced library
    and returns (event-timed ms per frame, trace [MAXCTA, TRACE_EV, 4] uint32 of
    the last frame).  Must run before anything loads the plain library."""
    import torch
    from . import q3tts, synth
    L = q3tts.load(build_traced())
    if not hasattr(L, "q3tts_trace_fetch"):
        raise RuntimeError("the plain library is already loaded in this process; trace in a fresh one")
    L.q3tts_trace_fetch.argtypes = [C.c_void_p, C.c_size_t]
    wl = synth.WORKLOADS[workload]
    s = wl.shape
    W = synth.make_weights(s, device="cuda")
    eng = q3tts.Engine(s, W, max_streams=1, kv_cap=wl.kv_cap, page_size=wl.page_size)
    eng.prefill(0, synth.make_prompts(s, [wl.prompt_lengths()[0]], device="cuda")[0])
    u = torch.from_numpy(synth.uniforms([0], frames)).cuda()
    codes = torch.zeros((1, 16), dtype=torch.int32, device="cuda")
    ev = []
    for f in range(frames):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(eng.stream)
        eng.step_frame([0], wl.sampling, u[:, f].contiguous(), codes)
        b.record(eng.stream)
        ev.append((a, b))
    eng.sync()
    ms = [a.elapsed_time(b) for a, b in ev]
    buf = np.zeros((MAXCTA * TRACE_EV, 4), dtype=np.uint32)
    if L.q3tts_trace_fetch(buf.ctypes.data, buf.nbytes) != 0:
        raise RuntimeError("q3tts_trace_fetch failed")
    eng.close()
    return ms, buf.reshape(MAXCTA, TRACE_EV, 4)


def step_kind(aux: int) -> str:
    k = KINDS[aux & 15]
    if (aux >> 4) & 31 == TALKER_PASS and (aux & 15) in (0, 2, 4):
        k += "_T"
    return k


def step_table(trace: np.ndarray, mhz: float = 2070.0) -> Dict[str, Tuple[float, float, float, float]]:
    """Per step kind: (occurrences per frame, median work us, median wait us,
    median longest ring wait of a warp us), over the CTAs that recorded steps.
    Times from clock64 (SM cycles at `mhz`)."""
    tag = (trace[:, :, 3] >> 16).astype(np.int64)
    aux = (trace[:, :, 3] & 0xFFFF).astype(np.int64)
    clk = trace[:, :, 2].astype(np.int64)
    work, wait, ring = (collections.defaultdict(list) for _ in range(3))
    ctas = 0
    for c in range(trace.shape[0]):
        n = int((tag[c] != 0).sum())
        steps = []  # [kind, start, arrival or None, ring wait of the step]
        for i in range(n):
            t, a, tm = int(tag[c, i]), int(aux[c, i]), int(clk[c, i])
            if t == TR_STEP:
                if a != FRAME_START:
                    steps.append([step_kind(a), tm, None, 0.0])
            elif t in (TR_ARRIVE, TR_END) and steps and steps[-1][2] is None:
                steps[-1][2] = tm
            elif t == TR_CW and steps:
                steps[-1][3] = a * 16 / mhz  # recorded before the next step starts
        if len(steps) < 2:
            continue
        ctas += 1
        for cur, nxt in zip(steps, steps[1:]):
            arr = cur[2] if cur[2] is not None else nxt[1]
            work[cur[0]].append((arr - cur[1]) / mhz)
            wait[cur[0]].append((nxt[1] - arr) / mhz)
            ring[cur[0]].append(cur[3])
    return {k: (len(work[k]) / max(ctas, 1), float(np.median(work[k])), float(np.median(wait[k])),
                float(np.median(ring[k]))) for k in work}


def barrier_table(trace: np.ndarray) -> Dict[str, Tuple[float, float, float, float]]:
    """Per kind of the step that a grid barrier ends ("START" for the frame's
    first): (barriers per frame, median arrival skew us -- the last CTA's
    arrival after the median CTA's --, median arrival spread us -- last minus
    first --, median release us -- from the last arrival to the first CTA
    that passes).  Times from the globaltimer, one clock for all SMs (ns);
    every CTA passes the same barriers in the same order."""
    tag = (trace[:, :, 3] >> 16).astype(np.int64)
    aux = (trace[:, :, 3] & 0xFFFF).astype(np.int64)
    g = trace[:, :, 0].astype(np.int64) | (trace[:, :, 1].astype(np.int64) << 32)
    arr, pas, kinds = [], [], None
    for c in range(trace.shape[0]):
        n = int((tag[c] != 0).sum())
        cur, a, p, k = None, [], [], []
        for i in range(n):
            t = int(tag[c, i])
            if t == TR_STEP:
                cur = "START" if aux[c, i] == FRAME_START else step_kind(int(aux[c, i]))
            elif t == TR_ARRIVE:
                a.append(int(g[c, i]))
                k.append(cur)
            elif t == TR_PASS:
                p.append(int(g[c, i]))
        if a:
            arr.append(a)
            pas.append(p)
            kinds = kinds or k
    if not arr:
        return {}
    nb = min(min(len(a) for a in arr), min(len(p) for p in pas))
    # nanoseconds since the epoch exceed float64's exact range: subtract a base first
    base = min(a[0] for a in arr)
    A = np.array([a[:nb] for a in arr], dtype=np.int64) - base
    P = np.array([p[:nb] for p in pas], dtype=np.int64) - base
    A, P = A.astype(np.float64), P.astype(np.float64)
    skew = (A.max(0) - np.median(A, 0)) / 1e3
    spread = (A.max(0) - A.min(0)) / 1e3
    release = (P.min(0) - A.max(0)) / 1e3
    out = {}
    for k in dict.fromkeys(kinds[:nb]):
        sel = np.array([kk == k for kk in kinds[:nb]])
        out[k] = (float(sel.sum()), float(np.median(skew[sel])), float(np.median(spread[sel])),
                  float(np.median(release[sel])))
    return out


def interval_table(trace: np.ndarray) -> Tuple[Dict[str, Tuple[int, float, float]], float]:
    """The frame split into barrier intervals, which add up to the whole frame:
    from one grid barrier's first pass (the frame's first step for the first
    interval) to the next barrier's last arrival -- the slowest CTA's work --
    plus that barrier's release to its first pass.  Intervals are keyed by the
    step kinds they hold, joined by "+", with (count, work us, release us)
    summed per key; the second value is the tail from the last barrier's first
    pass to the last CTA's end mark, us.  Globaltimer (ns), as barrier_table."""
    tag = (trace[:, :, 3] >> 16).astype(np.int64)
    aux = (trace[:, :, 3] & 0xFFFF).astype(np.int64)
    g = trace[:, :, 0].astype(np.int64) | (trace[:, :, 1].astype(np.int64) << 32)
    rows = []  # per CTA: (frame start, [(arrive, pass, step kinds)], end)
    for c in range(trace.shape[0]):
        n = int((tag[c] != 0).sum())
        start = end = arrive = None
        steps, bars = [], []
        for i in range(n):
            t, x, tm = int(tag[c, i]), int(aux[c, i]), int(g[c, i])
            if t == TR_STEP:
                if x == FRAME_START:
                    start = tm
                else:
                    steps.append(step_kind(x))
            elif t == TR_ARRIVE:
                arrive = tm
            elif t == TR_PASS:
                bars.append((arrive, tm, "+".join(steps)))
                steps = []
            elif t == TR_END:
                end = tm
        if start is not None:
            rows.append((start, bars, end))
    if not rows:
        return {}, 0.0
    nb = min(len(r[1]) for r in rows)
    prev = min(r[0] for r in rows)
    out: Dict[str, list] = {}
    for b in range(nb):
        last_arrival = max(r[1][b][0] for r in rows)
        first_pass = min(r[1][b][1] for r in rows)
        e = out.setdefault(rows[0][1][b][2], [0, 0.0, 0.0])
        e[0] += 1
        e[1] += (last_arrival - prev) / 1e3
        e[2] += (first_pass - last_arrival) / 1e3
        prev = first_pass
    ends = [r[2] for r in rows if r[2] is not None]
    tail = (max(ends) - prev) / 1e3 if ends else 0.0
    return {k: (v[0], v[1], v[2]) for k, v in out.items()}, tail


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", default="1.7b")
    ap.add_argument("--frames", type=int, default=12)
    args = ap.parse_args(argv)
    ms, trace = capture(args.workload, args.frames)
    print("traced frame ms:", [round(m, 3) for m in ms])
    table = step_table(trace)
    print("%-9s %6s %8s %8s %9s %10s" % ("step", "count", "work us", "wait us", "ring us", "total us"))
    for k, (n, w, q, r) in sorted(table.items(), key=lambda kv: -kv[1][0] * (kv[1][1] + kv[1][2])):
        print("%-9s %6.0f %8.2f %8.2f %9.2f %10.1f" % (k, n, w, q, r, n * (w + q)))
    intervals, tail = interval_table(trace)
    print("%-44s %6s %9s %10s" % ("interval (steps between barriers)", "count", "work us", "release us"))
    for k, (n, w, r) in sorted(intervals.items(), key=lambda kv: -(kv[1][1] + kv[1][2])):
        print("%-44s %6d %9.1f %10.1f" % (k[:44] or "(none)", n, w, r))
    print("%-44s %6s %9.1f" % ("tail after the last barrier", "", tail))
    print("%-9s %6s %8s %9s %10s" % ("barrier", "count", "skew us", "spread us", "release us"))
    for k, (n, sk, sp, rl) in barrier_table(trace).items():
        print("%-9s %6.0f %8.2f %9.2f %10.2f" % (k, n, sk, sp, rl))


if __name__ == "__main__":
    main()
