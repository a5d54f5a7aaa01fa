"""Multi-rank plumbing of bench.py on CPU (gloo, world_size 2).

The GEMV does not shard across GPUs in this build (replicas only): each rank
runs the whole workload and rank 0 reports the aggregate with the slowest
rank's time.  These tests cover that host-side logic without a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str) -> None:
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.rank_info() == (rank, world, rank)
        bench.barrier()
        # each rank reports a different time; every rank must see the slowest
        got = bench.max_over_ranks(1.5 + 10.0 * rank)
        bench.barrier()
        with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
            json.dump({"max": got}, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_barrier_with_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    for r in range(2):
        with open(tmp_path / f"rank{r}.json") as f:
            assert json.load(f)["max"] == pytest.approx(11.5)


def test_max_over_ranks_is_identity_without_a_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25) == 3.25
    bench.barrier()  # a no-op outside torch.distributed


def bench_host_cores():
    sys.path.insert(0, ROOT)
    import bench

    return bench.host_cores()


def _run_reference(env_extra):
    env = {**os.environ, **env_extra}
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                           "--warmup", "0"], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=300)


def test_reference_arm_prints_nothing_on_other_ranks():
    r = _run_reference({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    r = _run_reference({"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"})
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0 and line["higher_is_better"] is False
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"],
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert line["config"]["workload"] == "M16384_K8192_L16"
    assert line["cpu_baseline"]["cores"] == bench_host_cores()


def test_kernel_source_sets_cover_every_kernel_file():
    """Every source under csrc/ but the host planner, the repack and the wait
    self-test (no GEMV launch runs their code) belongs to some GEMV kernel's
    hash (so a changed kernel voids its recorded traffic)."""
    import os

    import bench

    csrc = os.path.join(bench.ROOT, "nvfp4_block_scaled_gemv_gb300", "csrc")
    files = set(os.listdir(csrc)) - {"api.cu", "repack.cu", "selftest.cu", "selftest.h"}
    listed = set().union(*bench.KERNEL_SOURCES.values())
    assert files == listed
    assert set(bench.KERNEL_SOURCES) == set(bench.KERNEL_NAMES)
    assert len({bench.kernel_source_hash(k) for k in bench.KERNEL_NAMES}) == len(bench.KERNEL_NAMES)
