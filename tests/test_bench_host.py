"""Host-side logic of bench.py, on CPU: multi-rank timing over gloo, the
whole-job throughput and roofline arithmetic, and the reference arm's
rank behaviour under a distributed launch."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, times, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        t = bench.max_over_ranks(times[rank], ws, torch.device("cpu"))
        v = bench.job_tflops(1e12, 10, t, ws)
        out.put((rank, t, v))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    ws, port = 2, _free_port()
    times = [12.5, 40.0]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, times, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(ws)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t, v in res:
        assert t == 40.0                      # every rank sees the slowest rank's time
        assert v == pytest.approx(2 * 1e12 * 10 / 0.040 / 1e12)  # all ranks' work / that time


def test_single_rank_is_identity():
    assert bench.max_over_ranks(3.0, 1, None) == 3.0
    assert bench.job_tflops(2e12, 5, 10.0, 1) == pytest.approx(1000.0)


def test_roofline_entry():
    # 0.5B projection, M = 8192: compute-bound at the measured peaks
    flops = 4 * 8192 * 4864 * 896
    nbytes = 2 * (8192 * 896 + 2 * 896 * 4864 + 8192 * 4864)
    r = bench.roofline_entry(flops, nbytes, 83.6, 1707.4, 6775.6)
    assert r["bound"] == "tensor"
    assert r["tflops"] == pytest.approx(flops / 83.6e-6 / 1e12)
    assert r["frac_of_roofline"] == pytest.approx((flops / 1707.4e12) / 83.6e-6)
    # M = 64: memory-bound
    flops = 4 * 64 * 4864 * 896
    nbytes = 2 * (64 * 896 + 2 * 896 * 4864 + 64 * 4864)
    r = bench.roofline_entry(flops, nbytes, 9.0, 1707.4, 6775.6)
    assert r["bound"] == "hbm"
    assert r["frac_of_roofline"] == pytest.approx((nbytes / 6775.6e9) / 9e-6)


def _run_bench(args, env_extra):
    env = dict(os.environ, **env_extra)
    env.setdefault("OMP_NUM_THREADS", "2")
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, env=env, timeout=300, cwd=ROOT)


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "0"],
                   {"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_rank0_prints_one_json_line():
    r = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "0",
                    "--workload", "qwen2.5-0.5b-m64", "--cpu-seconds", "1"],
                   {"WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"})
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 2
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["metric"] == bench.METRIC and d["higher_is_better"] is True
    # the same workload text as the library's arm prints for this workload
    assert d["config"]["workload"] == bench.describe_workload("qwen2.5-0.5b-m64")


def test_workload_descriptions_name_every_timed_form():
    for name, (K, N, Ms, seed) in bench.WORKLOADS.items():
        text = bench.describe_workload(name)
        assert text.startswith(name)
        assert f"K={K}" in text or f"H={K}" in text
        assert f"seed {seed}" in text and str(list(Ms)) in text
        if name.endswith(("-w4", "-mxfp8", "-nvfp4")):
            assert "K-major" in text
        elif not name.endswith("-mlp"):
            assert "interleaved" in text


def test_reference_arm_many_steps_sample_one_call_each():
    # a per-step budget below one all-call sample: each step samples one call
    # (in turn), so a long run stays bounded
    r = _run_bench(["--impl", "reference", "--steps", "12", "--warmup", "2",
                    "--workload", "qwen2.5-0.5b-m64", "--cpu-seconds", "0.001"],
                   {"WORLD_SIZE": "1", "RANK": "0", "LOCAL_RANK": "0"})
    assert r.returncode == 0, r.stderr
    d = json.loads([l for l in r.stdout.splitlines() if l.strip()][-1])
    assert d["steps"] == 12 and d["warmup"] == 2 and d["value"] > 0
    assert "steps of one call each" in d["cpu_baseline"]["sample"]
