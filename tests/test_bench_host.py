"""Host-side logic of bench.py, on CPU: the whole-job rate over replicas (the
slowest rank's time, reduced across two gloo ranks), the reference arm's
rank-0-only rule, and the guard that ties a recorded DRAM-traffic figure to
the frame kernel's code."""
import os
import shutil
import socket
import types

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, seconds, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, bench.slowest(seconds[rank], world, "cpu")))
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time_two_gloo_ranks():
    seconds = [1.25, 2.5]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, seconds, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 2.5, 1: 2.5}
    # 2 ranks x 16 streams x 10 steps over the slowest rank's 2.5 s
    assert bench.job_rate(160, 2, got[0]) == pytest.approx(128.0)


def test_single_rank_needs_no_process_group():
    assert bench.slowest(0.75, 1, "cpu") == 0.75
    assert bench.job_rate(200, 1, 0.5) == 400.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = types.SimpleNamespace(workload="1.7b", steps=1, warmup=0, gpus=2)
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""


def test_reference_arm_reports_the_workload_config(monkeypatch, capsys):
    """The reference arm (the oracle on the host, a bounded sample) prints one
    JSON line whose config is the workload's own -- the object the GPU arm
    prints -- and describes its sample in cpu_baseline."""
    import json
    from autoregressive_tts_decode_gb300 import synth
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    args = types.SimpleNamespace(workload="tiny", steps=1, warmup=0, gpus=1)
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["config"] == bench.workload_config(synth.WORKLOADS["tiny"], 1)
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0


def _sources():
    out = []
    for f in bench.KERNEL_SOURCES:
        with open(os.path.join(bench.ROOT, f), encoding="utf-8") as fh:
            out.append(fh.read())
    return out


def test_kernel_hash_follows_code_not_comments():
    texts = _sources()
    base = bench.kernel_source_sha(texts)
    assert base == bench.kernel_source_sha()
    commented = list(texts)
    commented[0] = "// a note\n" + texts[0].replace("\n", "  // trailing\n", 1) + "\n/* block\n comment */\n"
    assert bench.kernel_source_sha(commented) == base
    changed = list(texts)
    changed[1] = texts[1] + "\nconstexpr int unused_constant = 1;\n"
    assert bench.kernel_source_sha(changed) != base


def test_recorded_traffic_only_for_matching_code(tmp_path, monkeypatch):
    for f in bench.KERNEL_SOURCES:
        dst = tmp_path / f
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copy(os.path.join(bench.ROOT, f), dst)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_source_sha()
    prof = tmp_path / "profiles" / "frame_kernel_1p7b.md"
    prof.write_text('notes\n<!-- traffic {"sources_sha": "%s", "workload": "1.7b", '
                    '"dram_bytes_per_launch": 123} -->\n' % sha)
    assert bench.captured_traffic("1.7b") == 123.0
    assert bench.captured_traffic("0.6b") is None           # no capture for that workload
    src = tmp_path / bench.KERNEL_SOURCES[0]
    src.write_text(src.read_text() + "\n// comment only\n")
    assert bench.captured_traffic("1.7b") == 123.0
    src.write_text(src.read_text() + "\nconstexpr int changed = 2;\n")
    assert bench.captured_traffic("1.7b") is None           # the kernel changed since the capture


def test_nvtx_ranges_nest_without_a_device():
    """The bench's NVTX ranges (host timeline markers) open and close in order
    even on a machine without a GPU, and pass exceptions through."""
    import bench
    with bench.nvtx("outer"):
        with bench.nvtx("inner"):
            pass
    try:
        with bench.nvtx("raises"):
            raise ValueError("x")
    except ValueError:
        pass
