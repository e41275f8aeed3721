"""The benchmark's multi-rank host logic on CPU: two gloo ranks, as the
replicas-only N > 1 run launches them (one process per GPU there), and the
reference arm's rank rule (rank 0 alone works and prints)."""
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


def _rank_main(rank, world, port, out_path):
    import torch.distributed as dist

    sys.path.insert(0, ROOT)
    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank "measured" its own time; the slowest decides
        local = [0.25, 0.5][rank]
        dist.barrier()
        slowest = bench.max_over_ranks(local, world, device="cpu")
        value = bench.job_throughput(62, 10, world, slowest)
        with open(f"{out_path}.{rank}", "w") as f:
            json.dump({"slowest": slowest, "value": value}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time(tmp_path):
    torch = pytest.importorskip("torch")
    mp = torch.multiprocessing.get_context("spawn")
    port = _free_port()
    out = str(tmp_path / "res")
    procs = [mp.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = [json.load(open(f"{out}.{r}")) for r in range(2)]
    for r in res:
        assert r["slowest"] == 0.5
        # 62 tokens per step per rank, 10 steps, 2 ranks, 0.5 s
        assert r["value"] == pytest.approx(62 * 10 * 2 / 0.5)


def test_single_rank_passes_values_through():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.job_throughput(62, 4, 1, 2.0) == pytest.approx(124.0)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_runs_on_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
               CUDA_VISIBLE_DEVICES="")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                         env=env, timeout=600, cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    lines = [ln for ln in res.stdout.splitlines() if ln.strip()]
    if rank != 0:
        assert lines == []
        return
    line = json.loads(lines[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0


def test_all_cores_oracle_baseline_runs():
    # the spawn-started pool runs whole sweeps on every core, without CUDA
    sys.path.insert(0, ROOT)
    import bench

    res = bench.cpu_baseline_all_cores(seconds=1.0)
    assert res.get("error") is None, res
    assert res["kind"] == "oracle" and res["value"] > 0 and res["cores"] >= 1
    assert "one sweep per task" in res["sample"]
