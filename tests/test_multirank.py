"""The replicas-only multi-GPU path of bench.py, on CPU: two gloo ranks with different local
times agree on the slowest rank's time and on the whole-job value; the reference arm does its
work on rank 0 only."""

import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    local_ms = 100.0 + 50.0 * rank  # rank 1 is slower
    total = bench.slowest_rank_ms(local_ms)
    value = bench.whole_job_tflops(world, 10, 1e12, total)
    assert bench.dist_env() == (world, rank, rank)
    q.put((rank, total, value))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    out = sorted(q.get(timeout=10) for _ in range(world))
    for rank, total, value in out:
        assert total == 150.0
        # 2 replicas x 10 steps x 1 TFLOP in 0.15 s
        assert abs(value - 2 * 10 * 1e12 / 0.150 / 1e12) < 1e-9


def test_single_process_is_identity():
    import bench

    assert bench.slowest_rank_ms(12.5) == 12.5
    assert bench.whole_job_tflops(1, 4, 2e12, 8.0) == pytest.approx(1000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    import argparse

    import bench
    from fp16_gemm_relu_gb300 import workloads

    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(steps=3, warmup=3)
    assert bench.run_reference(args, workloads.get("square8192")) is None
    assert capsys.readouterr().out == ""


def test_traffic_rows_are_per_variant(tmp_path, monkeypatch):
    """A variant's run (int4 weights, another epilogue, the backward pass) never reads the DRAM
    bytes recorded for the plain forward relu GEMM of the same workload."""
    import bench

    assert bench.traffic_key("square8192", "forward", "relu", "none") == "square8192"
    assert bench.traffic_key("square8192", "forward", "relu", "w4") == "square8192/w4"
    assert (bench.traffic_key("square8192", "backward", "gelu", "none")
            == "square8192/backward/gelu")
    (tmp_path / "profiles").mkdir()
    h, hq = bench.kernel_source_hash(), bench.kernel_source_hash(dequant=True)
    assert h != hq  # the dequantising lines also hash the int4/NF4 kernels
    (tmp_path / "profiles" / "traffic.txt").write_text(
        f"# header\nsquare8192 {h} 100\nsquare8192/w4 {hq} 200\nsquare8192/nf4 {h} 250\n"
        f"skinny {h[::-1]} 300\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda dequant=False: hq if dequant else h)
    assert bench.traffic_from_profiles("square8192") == 100.0
    assert bench.traffic_from_profiles("square8192/w4") == 200.0
    assert bench.traffic_from_profiles("square8192/nf4") is None  # recorded with the dense hash
    assert bench.traffic_from_profiles("skinny") is None  # taken on another source


def test_oracle_sample_sizing_is_bounded():
    """The CPU-baseline leg and the reference arm size their oracle sample from a fixed plus
    per-row calibration; the sample stays within 1..M rows and grows with the time budget."""
    import bench
    from fp16_gemm_relu_gb300 import workloads

    wl = workloads.get("square256")
    a, b = wl.make_a(), wl.make_b()
    tiny = bench.sample_rows(wl, a, b, 1e-9)
    big = bench.sample_rows(wl, a, b, 1e3)
    assert tiny == 1
    assert big == wl.M
    assert 1 <= bench.sample_rows(wl, a, b, 0.05) <= wl.M
