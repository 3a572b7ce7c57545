"""Benchmark of the frame decode: acoustic frames/s (and RTF) on synthetic
weights of the named shapes, with the achieved HBM bandwidth of the frame step
against the measured roofline.

One step = one acoustic frame for every active stream of the workload (the
whole hot path: semantic draw, 15 CodePredictor passes with their draws, the
embedding sum and one Talker step).  Default workload: the 1.7B-class shapes at
batch 1 with Qwen-default sampling (prompt of 128 random embeddings, KV cap 512,
episodes of 240 frames per stream).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica (the decode has
no exchange step); value = frames of all ranks / max-over-ranks time.
`--impl reference` times the CPU oracle on the same workload (bounded samples).
"""
from __future__ import annotations

import argparse
import contextlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "acoustic frames/sec (RTF) at batch 1 and batched; achieved HBM GB/s vs roofline"
UNIT = "frames/s"


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def slowest(seconds, world, device):
    """The largest of the ranks' timed-region lengths (every rank gets it): the
    whole job's time, since the replicas run side by side.  One rank: itself."""
    if world <= 1:
        return float(seconds)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(seconds)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(frames_per_rank, world, seconds):
    """Whole-job throughput: the frames all ranks decoded over the slowest
    rank's time."""
    return frames_per_rank * world / seconds


# Sources of the persistent frame kernel: a recorded DRAM-traffic figure holds
# only for the code it was captured from.
# (The handle's host-side struct in engine.cuh is not among them: its fields
# do not reach the kernel's device code.)
KERNEL_SOURCES = ("autoregressive_tts_decode_gb300/csrc/frame_kernel.cu",
                  "autoregressive_tts_decode_gb300/csrc/sampler.cuh",
                  "autoregressive_tts_decode_gb300/csrc/common.cuh", "include/q3tts.h")


def _code_only(text):
    """C/C++ source without comments and blank lines: edits to comments do not
    change what is compiled (these sources hold no string literal with a
    comment marker)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.rstrip() for line in text.splitlines() if line.strip())


def kernel_source_sha(texts=None):
    """Hash of the frame kernel's code (comments excluded); `texts` overrides
    the files' contents (same order as KERNEL_SOURCES)."""
    import hashlib
    h = hashlib.sha256()
    for i, f in enumerate(KERNEL_SOURCES):
        if texts is None:
            with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
                t = fh.read()
        else:
            t = texts[i]
        h.update(_code_only(t).encode("utf-8"))
    return h.hexdigest()[:16]


def captured_traffic(workload):
    """DRAM bytes (read + write) per frame-kernel launch from the ncu capture
    summarised in profiles/frame_kernel_<workload>.md (its `traffic` marker),
    or None if that capture was of other kernel sources or is missing."""
    p = os.path.join(ROOT, "profiles", "frame_kernel_%s.md" % workload.replace(".", "p"))
    if not os.path.exists(p):
        return None
    with open(p) as f:
        for line in f:
            if line.startswith("<!-- traffic "):
                d = json.loads(line[len("<!-- traffic "):].rsplit("-->", 1)[0])
                if d.get("sources_sha") == kernel_source_sha() and d.get("workload") == workload:
                    return float(d["dram_bytes_per_launch"])
    return None


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.rows.append(parts)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in self.rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="1.7b")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-ttfa", action="store_true", help="skip the prefill / first-frame timing")
    return ap.parse_args()


def episode_plan(wl, total_frames):
    """Streams needed so that each runs at most wl.frames frames after its prompt."""
    per = wl.frames
    return max(1, math.ceil(total_frames / per))


def cpu_baseline(wl, sample_frames=3, prompt_len=16):
    """Times the CPU oracle (as it stands) for a few frames of the workload's shapes
    after a short prompt; returns frames/s and the sample description."""
    import torch
    from autoregressive_tts_decode_gb300 import synth
    from oracle import oracle
    s = wl.shape
    W = synth.make_weights(s, device="cuda")
    Wc = {k: v.cpu() for k, v in W.items()}
    del W
    torch.cuda.empty_cache()
    orc = oracle.Oracle(s, Wc, 1, wl.kv_cap)
    orc.prefill(0, synth.make_prompts(s, [prompt_len])[0].numpy())
    u = synth.uniforms([0], sample_frames + 3)[0]
    orc.step_frame(0, wl.sampling, u[0])  # warm-up
    cores = oracle.max_threads()
    t0 = time.perf_counter()
    for f in range(sample_frames):
        orc.step_frame(0, wl.sampling, u[f + 1])
    dt = time.perf_counter() - t0
    # the same oracle on one core, for two further frames
    oracle.set_threads(1)
    t1 = time.perf_counter()
    for f in range(2):
        orc.step_frame(0, wl.sampling, u[sample_frames + 1 + f])
    dt1 = time.perf_counter() - t1
    oracle.set_threads(cores)
    return {"value": sample_frames / dt, "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"{sample_frames} frames of stream 0 after a {prompt_len}-position prompt "
                      f"(one warm-up frame discarded), {wl.name} shapes, fp64 oracle",
            "one_core": {"value": 2 / dt1, "unit": UNIT, "cores": 1,
                         "sample": "the next 2 frames of the same stream on one thread"}}


@contextlib.contextmanager
def nvtx(name):
    """A named NVTX range on the host timeline (prefill, warm-up, timed frames,
    end-to-end frames, each frame), for timeline tools; it adds host work only."""
    import torch
    torch.cuda.nvtx.range_push(name)
    try:
        yield
    finally:
        torch.cuda.nvtx.range_pop()


def prefill_and_ttfa(eng, stream, prompt, sampling, u_dev, codes, reps=5):
    """Prefill time of one prompt and the time to the first frame of codes.

    Device-timed: CUDA events on the engine's stream around q3tts_prefill alone,
    and around prefill + the first frame decode (codes on the device).  End to
    end: from the host's pinned prompt to the first frame's 16 codes back in
    pinned host memory (H2D copy, prefill, frame, D2H copy, synchronise).  The
    codec decoder that turns codes into samples is not part of this library, so
    first audio here means the first frame of codes.  Median of `reps` runs
    after one warm-up run."""
    import torch
    st = eng.stream
    host_p = prompt.cpu().pin_memory()
    dev_p = torch.empty_like(prompt)
    host_c = torch.zeros((1, 16), dtype=torch.int32).pin_memory()
    pre, ttfa, e2e = [], [], []
    for r in range(reps + 1):
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        torch.cuda.synchronize()
        a.record(st)
        with nvtx("prefill"):
            eng.prefill(stream, prompt)
        b.record(st)
        with nvtx("first frame"):
            eng.step_frame([stream], sampling, u_dev, codes)
        c.record(st)
        eng.sync()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dev_p.copy_(host_p, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        eng.prefill(stream, dev_p)
        eng.step_frame([stream], sampling, u_dev, codes)
        host_c.copy_(codes[:1], non_blocking=True)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        if r:
            pre.append(a.elapsed_time(b))
            ttfa.append(a.elapsed_time(c))
            e2e.append(1e3 * dt)
    L = int(prompt.shape[0])
    med = statistics.median
    return {"prompt_len": L, "prefill_ms": med(pre), "prefill_tokens_per_s": 1e3 * L / med(pre),
            "ttfa_ms": med(ttfa), "ttfa_e2e_ms": med(e2e), "runs": reps,
            "note": "first audio = first frame of 16 codes (prefill + one frame decode); "
                    "excluded from frames/s"}


def streaming_chunks(eng, stream, prompt, sampling, uni_dev, frames=64, chunks=(1, 8, 32)):
    """Frame-incremental decode through q3tts_step_frames (double-buffered, codes to
    pinned host memory): per chunk size, the host time from a finished prefill
    to the first chunk's codes on the host, and frames/s over `frames` frames."""
    import torch
    out = {}
    u = uni_dev[:frames].unsqueeze(1).contiguous()  # [frames, 1, 16]
    for ch in chunks:
        eng.prefill(stream, prompt)
        eng.sync()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        first = None
        n = 0
        for c in eng.stream_codes([stream], sampling, u, ch):
            if first is None:
                first = time.perf_counter() - t0
            n += c.shape[0]
        dt = time.perf_counter() - t0
        out[str(ch)] = {"first_chunk_ms": 1e3 * first, "frames_per_s": n / dt}
    return {"frames": frames, "chunks": out,
            "note": "host-timed: prefill done -> codes in pinned host memory; chunk k+1 is "
                    "enqueued before the host waits for chunk k"}


L2_BYTES = 129e6  # GB300 L2


def workload_config(wl, world):
    """The `config` object of a bench line: the workload as both arms run it."""
    from autoregressive_tts_decode_gb300 import bytes_model, synth
    s = wl.shape
    lens = wl.prompt_lengths()
    B = wl.streams
    fb = bytes_model.frame_bytes(s, lens[0])
    weights = fb.talker_weights + (synth.N_CODEBOOKS - 1) * fb.cp_pass_weights
    return {"workload": wl.name, "streams_per_gpu": B,
            "prompt_len": lens if B > 1 else lens[0], "kv_cap": wl.kv_cap,
            "page_size": wl.page_size,
            "kv_cache": {synth.DTYPE_F32: "fp32", synth.DTYPE_BF16: "bf16"}.get(s.kv_dtype, "?"),
            "frames_per_episode": wl.frames,
            "sampling": "greedy" if not wl.sampling.do_sample else "top_k50_T0.9_rep1.05",
            "parallelism": f"replicas x{world}",
            "l2": ("inputs larger than L2: each step streams %.2f GB of weights" if weights > L2_BYTES
                   else "inputs within L2 (%.2f GB of weights per step): not an L2-cold figure") % (weights / 1e9)}


def run_reference(args):
    """The reference arm: the CPU oracle on this workload, bounded per step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from autoregressive_tts_decode_gb300 import synth
    import torch
    from oracle import oracle
    wl = synth.WORKLOADS[args.workload]
    s = wl.shape
    W = synth.make_weights(s, device="cuda" if torch.cuda.is_available() else "cpu")
    Wc = {k: v.cpu() for k, v in W.items()}
    del W
    orc = oracle.Oracle(s, Wc, 1, wl.kv_cap)
    orc.prefill(0, synth.make_prompts(s, [16])[0].numpy())
    steps = max(1, min(args.steps, 8))
    warm = max(0, min(args.warmup, 1))
    u = synth.uniforms([0], steps + warm)[0]
    for f in range(warm):
        orc.step_frame(0, wl.sampling, u[f])
    t0 = time.perf_counter()
    for f in range(steps):
        orc.step_frame(0, wl.sampling, u[warm + f])
    dt = time.perf_counter() - t0
    v = steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": steps, "warmup": warm, "ms_per_step": 1e3 * dt / steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "rtf": synth.FRAMES_PER_SECOND / v,
            "config": workload_config(wl, world),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": oracle.max_threads(),
                             "kind": "oracle",
                             "sample": f"{steps} frames of one stream after a 16-position prompt "
                                       f"(oracle steps capped at 8 to bound CPU time; the workload's own "
                                       f"prompt and streams are in config)"},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
        return
    import numpy as np
    import torch
    import torch.distributed as dist

    from autoregressive_tts_decode_gb300 import build, bytes_model, q3tts, synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build.build()
    wl = synth.WORKLOADS[args.workload]
    s = wl.shape
    B = wl.streams
    total = args.warmup + args.steps
    episodes = episode_plan(wl, total)
    n_streams = B * episodes
    W = synth.make_weights(s, device="cuda")
    lens = wl.prompt_lengths()
    torch.cuda.synchronize()
    eng = q3tts.Engine(s, W, max_streams=n_streams, kv_cap=wl.kv_cap, page_size=wl.page_size)
    # every episode's streams get their prompts before timing
    prompts = synth.make_prompts(s, lens, device="cuda")
    with nvtx("prefill"):
        for e in range(episodes):
            for b in range(B):
                eng.prefill(e * B + b, prompts[b])
        torch.cuda.synchronize()
    uni = synth.uniforms(list(range(n_streams)), wl.frames)  # [streams, frames, 16]
    uni_d = torch.from_numpy(uni).to("cuda")
    codes = torch.zeros((B, 16), dtype=torch.int32, device="cuda")
    frames_run = [0] * episodes

    def plan(step):
        e = min(step // wl.frames, episodes - 1)
        f = frames_run[e]
        frames_run[e] += 1
        ids = [e * B + b for b in range(B)]
        return ids, f

    def step_args(step):
        ids, f = plan(step)
        u = uni_d[ids[0]:ids[-1] + 1, f].contiguous()
        return ids, u

    stream = eng.stream
    with nvtx("warm-up"):
        for i in range(args.warmup):
            ids, u = step_args(i)
            eng.step_frame(ids, wl.sampling, u, codes)
        eng.sync()
    # pre-build each step's uniforms so the timed loop does no host work
    pre = [step_args(args.warmup + i) for i in range(args.steps)]
    launches0 = eng.kernel_launches()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        t_start.record(stream)
        with nvtx("timed frames"):
            for i in range(args.steps):
                ids, u = pre[i]
                ev[i][0].record(stream)
                with nvtx("frame"):
                    eng.step_frame(ids, wl.sampling, u, codes)
                ev[i][1].record(stream)
            t_end.record(stream)
            torch.cuda.synchronize()
    eng.sync()
    launches = eng.kernel_launches() - launches0
    elapsed = t_start.elapsed_time(t_end) / 1e3
    step_ms = [a.elapsed_time(b) for a, b in ev]
    elapsed = slowest(elapsed, world, "cuda")
    value = job_rate(args.steps * B, world, elapsed)

    # algorithmic bytes of the timed steps (weights once per use, KV per stream)
    byts = 0
    fr = [0] * episodes
    for i in range(args.warmup + args.steps):
        e = min(i // wl.frames, episodes - 1)
        if i >= args.warmup:
            pos = [lens[b] + fr[e] for b in range(B)]
            byts += (bytes_model.frame_bytes(s, pos[0]).total if B == 1
                     else bytes_model.batched_step_bytes(s, pos))
        fr[e] += 1
    bytes_per_step = byts / args.steps
    mean_step = statistics.mean(step_ms) / 1e3
    peak, peak_kind = measured_peaks()
    achieved = bytes_per_step / mean_step / 1e9
    clocks = clk.summary()

    # end to end through the public API: per step, upload that step's uniforms
    # from pinned host memory and read the codes back before the next step.
    e2e = None
    if not args.no_e2e:
        eng.reset(-1)
        for e in range(episodes):
            for b in range(B):
                eng.prefill(e * B + b, prompts[b])
        frames_run[:] = [0] * episodes
        host_u = torch.from_numpy(uni).pin_memory()
        host_codes = torch.zeros((B, 16), dtype=torch.int32).pin_memory()
        dev_u = torch.zeros((B, 16), dtype=torch.float32, device="cuda")
        for i in range(args.warmup):
            ids, f = plan(i)
            dev_u.copy_(host_u[ids[0]:ids[-1] + 1, f], non_blocking=True)
            eng.step_frame(ids, wl.sampling, dev_u, codes)
            host_codes.copy_(codes, non_blocking=True)
            torch.cuda.current_stream().synchronize()
        eng.sync()
        plans = [plan(args.warmup + i) for i in range(args.steps)]
        srcs = [host_u[ids[0]:ids[-1] + 1, f] for ids, f in plans]
        torch.cuda.synchronize()
        with nvtx("end-to-end frames"):
            t0 = time.perf_counter()
            for i in range(args.steps):
                ids, f = plans[i]
                dev_u.copy_(srcs[i], non_blocking=True)
                eng.step_frame(ids, wl.sampling, dev_u, codes)
                host_codes.copy_(codes, non_blocking=True)
                torch.cuda.current_stream().synchronize()
            dt = time.perf_counter() - t0
        eng.sync()
        dt = slowest(dt, world, "cuda")
        e2e = {"value": job_rate(args.steps * B, world, dt), "unit": UNIT,
               "h2d_bytes_per_step": 16 * 4 * B,
               "d2h_bytes_per_step": 16 * 4 * B}

    ttfa = prefill_and_ttfa(eng, 0, prompts[0], wl.sampling, uni_d[0:1, 0].contiguous(),
                            codes) if rank == 0 and not args.no_ttfa else None
    streaming = (streaming_chunks(eng, 0, prompts[0], wl.sampling, uni_d[0])
                 if rank == 0 and not args.no_ttfa and wl.kv_cap - lens[0] > 64 else None)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        eng.close()
        del W
        torch.cuda.empty_cache()
        cpu = cpu_baseline(wl)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * elapsed / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": {synth.DTYPE_BF16: "bf16", synth.DTYPE_FP8: "fp8-e4m3 weights"}.get(s.weight_dtype, "f32"),
            "data": "synthetic (random N(0,0.02) weights of the named shapes, N(0,1) prompts, "
                    "seeded uniforms)",
            "rtf": synth.FRAMES_PER_SECOND / (value / world),
            "config": workload_config(wl, world),
            "roofline": {"bound": "hbm",
                         "kernel": ("frame_kernel (persistent, one launch per frame)"
                                    if launches == args.steps else
                                    "frame step (all launches of one frame)"),
                         "achieved": achieved, "peak": peak, "peak_kind": peak_kind,
                         "unit": "GB/s", "frac": achieved / peak,
                         "traffic": captured_traffic(wl.name) if launches == args.steps else None,
                         "algorithmic_bytes_per_step": bytes_per_step,
                         "step_ms_median": statistics.median(step_ms),
                         "step_ms_p90": sorted(step_ms)[int(0.9 * (len(step_ms) - 1))]},
            "prefill": ttfa,
            "streaming": streaming,
            "gpu_launches": launches,
            "clocks": clocks,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "memory": {"peak_allocated_gb": torch.cuda.max_memory_allocated() / 1e9,
                       "peak_reserved_gb": torch.cuda.max_memory_reserved() / 1e9},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
