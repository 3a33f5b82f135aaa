"""bench.py's host logic without a GPU: the multi-rank helpers on two gloo
ranks, the weak-scaling aggregate, and the reference (oracle) arm's JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.dist_env()
        bench.barrier(w)
        t = bench.max_over_ranks(1.0 + rank, w, torch.device("cpu"))
        q.put((r, w, lr, t, bench.shard_seed(2, r)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(world))
    assert [g[0] for g in got] == [0, 1] and all(g[1] == 2 for g in got)
    assert all(g[3] == 2.0 for g in got)          # max over ranks
    assert got[0][4] != got[1][4]                 # each rank draws its own batch


def test_weak_scaling_aggregate():
    # 2 ranks x 10 steps x 1e12 FLOP in 4 s -> 5 TFLOP/s for the job
    assert bench.job_throughput(1e12, 10, 2, 4.0) == pytest.approx(5.0)
    assert bench.job_throughput(1e12, 10, 1, 4.0) == pytest.approx(2.5)


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl",
                        "reference", "--steps", "2", "--warmup", "0",
                        "--ref-seconds", "1", "--workload", "pr1_B1H1S128D64_fp16"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl",
                        "reference", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_kernel_fingerprint_covers_device_code_only(tmp_path, monkeypatch):
    """The fingerprint that keys the committed ncu traffic records changes with
    the device code and launch wrappers, not with the host-side dispatch."""
    import shutil
    src = os.path.join(ROOT, "attention_forward_gb300", "csrc")
    dst = tmp_path / "attention_forward_gb300" / "csrc"
    shutil.copytree(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    f0 = bench.kernel_fingerprint()
    assert f0 == bench.kernel_fingerprint()
    api = dst / "fa_api.cu"
    api.write_text(api.read_text() + "\n// a host-side edit\n")
    assert bench.kernel_fingerprint() == f0
    dev = dst / "fa_prefill_pair.cuh"
    dev.write_text(dev.read_text() + "\n// a comment changes no kernel\n")
    assert bench.kernel_fingerprint() == f0
    dev.write_text(dev.read_text() + "\nconstexpr int kDeviceSideEdit = 1;\n")
    assert bench.kernel_fingerprint() != f0


def test_paired_summary_margins_and_halves():
    """margin = t_A / t_B per alternation; its median, the AB and BA halves
    and B's wins; B 2 % faster in every alternation gives margin 1/0.98."""
    res = [(1.0, 0.98, "AB" if i % 2 == 0 else "BA") for i in range(10)]
    d = bench.paired_summary(res)
    assert d["margin"] == pytest.approx(1 / 0.98)
    assert d["ab_half"] == pytest.approx(1 / 0.98) and d["ba_half"] == pytest.approx(1 / 0.98)
    assert d["b_wins"] == 10 and d["alternations"] == 10
    # an order effect shows in the halves, not in the median of both
    res = [(1.0, 0.99, "AB"), (1.0, 1.01, "BA")] * 5
    d = bench.paired_summary(res)
    assert d["ab_half"] > 1 > d["ba_half"] and d["b_wins"] == 5


def test_aa_noise_is_the_p95_of_the_deviation():
    t, mx = bench.aa_noise([1.0, 1.001, 0.999, 1.0, 1.0, 1.0005, 0.9998, 1.0, 1.0, 0.997])
    assert mx == pytest.approx(0.003)
    assert 0.001 <= t <= 0.003


def test_clock_summary_counts_only_samples_inside_the_region():
    """Clock samples outside the timed region are never used, and a region
    with fewer than three samples is marked."""
    c = bench.NvmlClocks.__new__(bench.NvmlClocks)
    c.ok, c.max_mhz = True, 2070.0
    c.samples = [(0.5, 1000.0, 150.0, 0), (1.1, 1980.0, 900.0, 0x4),
                 (1.2, 1995.0, 950.0, 0), (1.3, 2010.0, 980.0, 0), (9.0, 900.0, 100.0, 0x8)]
    d = c.summary(1.0, 2.0)
    assert d["samples"] == 3 and d["sm_mhz"] == 1995.0 and d["sm_mhz_min"] == 1980.0
    assert d["reasons"] == ["sw_power_cap"] and "note" not in d
    d = c.summary(1.15, 1.25)
    assert d["samples"] == 1 and "fewer than 3" in d["note"]
    d = c.summary(3.0, 4.0)
    assert d["samples"] == 0 and d["sm_mhz"] is None
