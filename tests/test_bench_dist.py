"""Host-side logic of the benchmark's multi-process path, on CPU with gloo and two ranks:
process-group setup from the torchrun environment, the barrier, the max over ranks of the step
time, the whole-job (weak-scaling) throughput, and the reference arm's rank-0-only rule."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, q):
    try:
        sys.path.insert(0, ROOT)
        os.environ.update(WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                          MASTER_PORT=str(port))
        import bench
        import torch.distributed as dist
        world, r, local = bench.dist_setup(backend="gloo")
        bench.barrier(world)
        # rank 0 took 2.0 ms per step, rank 1 took 3.0 ms: the job's step is the slower one
        step_ms = bench.max_over_ranks(2.0 + r, world)
        rate = bench.job_throughput(16384, world, step_ms)

        class A:
            steps, warmup = 1, 0
        ref = bench.run_reference(A(), world, r) if r == 1 else "skipped"
        dist.destroy_process_group()
        q.put((r, world, local, step_ms, rate, ref))
    except Exception as e:  # report instead of hanging the parent
        q.put(("error", repr(e)))


def test_two_rank_gloo_timing_and_throughput():
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(r[0] != "error" for r in res), res
    res.sort()
    for r, world, local, step_ms, rate, ref in res:
        assert world == 2 and local == r
        assert step_ms == 3.0                                   # max over ranks
        assert rate == pytest.approx(16384 * 2 / 3.0e-3)        # all ranks' tokens / slowest step
    assert res[1][5] is None                                    # reference arm: rank 1 does no work


def test_single_process_defaults():
    sys.path.insert(0, ROOT)
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_setup() == (1, 0, 0)
    assert bench.max_over_ranks(1.25, 1) == 1.25
    assert bench.job_throughput(100, 1, 10.0) == pytest.approx(1e4)


def test_gemm_traffic_is_reported_only_for_the_profiled_source(tmp_path, monkeypatch):
    """roofline.traffic comes from the committed ncu summary while gemm.cu is the source those
    counters were taken on (SHA-256 recorded beside them), and is None once it differs."""
    import hashlib

    import bench
    src = tmp_path / "gemm.cu"
    src.write_text("kernel v1")
    sha = hashlib.sha256(b"kernel v1").hexdigest()
    prof = tmp_path / "traffic.md"
    prof.write_text(f"traffic: launch=gate_up dram_read=100 dram_write=23 gemm_cu_sha256={sha}\n"
                    f"traffic: launch=down dram_read=7 dram_write=8 gemm_cu_sha256={sha}\n")
    monkeypatch.setattr(bench, "GEMM_SOURCE", str(src))
    monkeypatch.setattr(bench, "TRAFFIC_PROFILE", str(prof))
    assert bench.gemm_traffic_per_launch("gate_up") == 123
    assert bench.gemm_traffic_per_launch("down") == 15
    assert bench.gemm_traffic_per_launch("other") is None
    src.write_text("kernel v2")
    assert bench.gemm_traffic_per_launch("gate_up") is None

