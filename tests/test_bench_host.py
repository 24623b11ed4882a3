"""Host-side logic of bench.py without a GPU: the max-over-ranks reduction under a
real 2-rank gloo process group, the rank-0-only reference arm, and the parser of the
nvidia-smi clock samples."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    bench.init_dist(world, "gloo")
    bench.barrier()
    got = bench.reduce_max(1.5 + rank)  # rank 0 reports 1.5, rank 1 reports 2.5
    out[rank] = got
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_reduce_max_without_a_process_group_is_identity():
    assert bench.reduce_max(3.25) == 3.25


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_reference_arm_prints_one_json_line(tmp_path):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "3",
                        "--warmup", "3", "--workload", "per_row_256x512x512"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TOPS" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["config"]["workload"] == "per_row_256x512x512"


def test_clock_sample_parser():
    lines = [
        "0, 2070, 2070, 1012.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 1950, 2070, 1390.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2010, 2070, 1201.0, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    c = bench.ClockSampler.parse(lines)
    assert c == {"sm_mhz": 2010.0, "sm_max_mhz": 2070.0, "samples": 3, "reasons": ["sw_power_cap"]}
    assert bench.ClockSampler.parse([]) is None


def test_profiled_traffic_is_null_for_another_workload():
    assert bench.profiled_traffic("no_such_workload") is None


def test_committed_profile_records():
    """The GEMM traffic record is for the bench default (reported only while it hashes the
    current GEMM sources); the int8 rate record names its instruction and its summary."""
    d = json.load(open(bench.PROFILE_TRAFFIC))["gemm"]
    assert d["workload"] == bench.DEFAULT_WORKLOAD and d["dram_bytes_per_launch"] > 0
    assert bench.profiled_traffic(bench.DEFAULT_WORKLOAD) in (None, d["dram_bytes_per_launch"])
    i8 = bench.int8_dense_peak()
    assert i8 is not None and i8["value"] > 0 and "mma.sync" in i8["instruction"]
    assert os.path.exists(os.path.join(ROOT, i8["from"]))


def test_profiled_traffic_is_null_once_the_gemm_source_changes(monkeypatch):
    monkeypatch.setattr(bench, "GEMM_SOURCES", bench.GEMM_SOURCES + ["bench.py"])
    assert bench.profiled_traffic(bench.DEFAULT_WORKLOAD) is None
