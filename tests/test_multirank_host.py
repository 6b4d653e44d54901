"""Host logic of the multi-GPU bench path, run as two gloo ranks on the CPU.

With N GPUs the bench runs N independent problems (one per rank, no
collective on the data path); the only cross-rank steps are a barrier around
the timed region and a max-reduction of the times.  These tests run exactly
those helpers from bench.py in two processes.
"""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import mca_inputs


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out_dir: str):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cpu = torch.device("cpu")
        w = mca_inputs.WORKLOADS["tiny_causal_f32"]
        seed = bench.rank_seed(mca_inputs.WORKLOAD_ORDER.index(w.name) + 1, rank)
        Z = mca_inputs.workload_inputs(w, seed)[0]
        bench.barrier()
        # each rank's own elapsed time; the job's time is the slowest one
        local_s = 0.25 + 0.5 * rank
        max_s = bench.reduce_max(local_s, cpu)
        rate = bench.whole_job_rate(world, w.B * w.n, 7, max_s)
        bench.barrier()
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump({"seed": seed, "max_s": max_s, "rate": rate,
                       "z_sum": float(Z.double().sum()), "z0": float(Z.flatten()[0])}, f)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(180)
def test_two_ranks_time_rate_and_inputs(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    r = [json.load(open(tmp_path / f"r{k}.json")) for k in range(world)]
    w = mca_inputs.WORKLOADS["tiny_causal_f32"]
    # both ranks agree on the slowest rank's time
    assert r[0]["max_s"] == r[1]["max_s"] == pytest.approx(0.75)
    # whole-job rate: every rank's tokens over the slowest time
    assert r[0]["rate"] == pytest.approx(world * w.B * w.n * 7 / 0.75)
    assert r[0]["rate"] == r[1]["rate"]
    # rank 0 runs the workload's own problem; the other rank a different one
    assert r[0]["seed"] == mca_inputs.WORKLOAD_ORDER.index(w.name) + 1
    assert r[1]["seed"] != r[0]["seed"]
    assert r[0]["z_sum"] != r[1]["z_sum"] and r[0]["z0"] != r[1]["z0"]


def test_single_process_helpers_are_identity():
    assert bench.reduce_max(3.5, torch.device("cpu")) == 3.5
    bench.barrier()  # no process group: a no-op
    assert bench.whole_job_rate(1, 100, 10, 2.0) == 500.0
    assert bench.rank_seed(4, 0) == 4


def _scan_worker(rank: int, world: int, port: int, out_dir: str):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from flash_mixed_chunk_gb300.seqsplit import exclusive_state_scan
        g = torch.Generator().manual_seed(100 + rank)
        local = torch.randn(2, 3, 4, generator=g, dtype=torch.float32)
        state_in = exclusive_state_scan(local)
        torch.save({"local": local, "state_in": state_in}, os.path.join(out_dir, f"s{rank}.pt"))
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(180)
@pytest.mark.parametrize("world", [2, 3])
def test_exclusive_state_scan_over_ranks(tmp_path, world):
    """The carried-in state of a sequence split over ranks: rank r receives the
    sum of the per-rank state sums of ranks 0 .. r-1 (zeros on rank 0)."""
    mp.start_processes(_scan_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = [torch.load(tmp_path / f"s{k}.pt") for k in range(world)]
    run = torch.zeros(2, 3, 4)
    for k in range(world):
        assert torch.equal(got[k]["state_in"], run)
        run = run + got[k]["local"]
