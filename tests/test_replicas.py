"""N > 1 on CPU: the replica bookkeeping of bench.py over a world-size-2 gloo group.

The layer does not shard (one process per GPU runs an independent replica), so the only
multi-process logic is the timing barrier, the max over ranks of the timed region and the
whole-job value; these run here on gloo with two ranks.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, ms_by_rank, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, wsz, local = bench.dist_env()
        bench.dist_barrier(wsz)
        ms_max = bench.dist_max(ms_by_rank[rank], wsz)
        value = bench.job_value(wsz, 64, 10, ms_max)
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as fh:
            json.dump({"rank": r, "world": wsz, "local": local, "ms_max": ms_max, "value": value}, fh)
    finally:
        dist.destroy_process_group()


def test_replica_max_and_job_value(tmp_path):
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    ms = [120.0, 150.0]
    mp.spawn(_worker, args=(world, port, ms, str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    for r, d in enumerate(res):
        assert d["rank"] == r and d["world"] == world and d["local"] == r
        assert d["ms_max"] == max(ms)                      # every rank sees the slowest replica
        # whole-job tokens/s: 2 replicas x 64 tokens x 10 steps over the slowest time
        assert d["value"] == pytest.approx(world * 64 * 10 / (max(ms) / 1000.0))


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_max(3.5, 1) == 3.5
    bench.dist_barrier(1)
    assert bench.job_value(1, 1, 1, 1000.0) == pytest.approx(1.0)


def test_reference_arm_other_ranks_exit_quietly():
    """Under torchrun only rank 0 runs and prints the oracle line; other ranks exit 0."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


@pytest.mark.parametrize("workload", ["tiny", "full_tiny"])
def test_reference_arm_line(workload):
    """Rank 0 of the reference arm times the oracle and prints one JSON line with the
    contract's keys, its cpu_baseline and a zero-copy e2e."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", workload, "--steps", "2", "--warmup", "1", "--cpu-budget-s", "0.5"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["config"]["workload"] == workload
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_two_workloads():
    """A list of workloads gives one line: the first workload's record at the top level and
    each other one's complete record under its own name (the default is the headline pair
    decode_t1,prefill_t4096)."""
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny,full_tiny", "--steps", "1", "--warmup", "0",
                        "--cpu-budget-s", "0.2"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["config"]["workload"] == "tiny" and line["value"] > 0
    sub = line["full_tiny"]
    assert sub["config"]["workload"] == "full_tiny" and sub["value"] > 0
    for key in ("value", "unit", "ms_per_step", "cpu_baseline", "e2e", "config"):
        assert key in sub, key
    sys.path.insert(0, ROOT)
    import bench
    assert bench.DEFAULT_WORKLOADS.split(",") == ["decode_t1", "prefill_t4096"]


def test_workload_list_keeps_overrides_together():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.workload_specs("decode_t1,prefill_t4096") == ["decode_t1", "prefill_t4096"]
    assert bench.workload_specs("prefill_t4096:E=128,T=600") == ["prefill_t4096:E=128,T=600"]
    assert bench.workload_specs("full_t1:E=64,decode_t1:T=4") == ["full_t1:E=64", "decode_t1:T=4"]
