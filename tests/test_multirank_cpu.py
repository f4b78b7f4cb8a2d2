"""The benchmark's N > 1 path on CPU with world size 2 over gloo: each rank runs an
independent layer on its own batch (no collective on the data path); the job's step
time is the slowest rank's and its throughput counts every rank's tokens."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import workloads
    ms = [3.0, 5.0][rank]
    got = bench.slowest_rank_ms(ms, dist, torch.device("cpu"))
    # the ranks' batches differ (one seed per rank), as in the benchmark
    shape = workloads.LayerShape("t", N=16, H=16, I=16, E=4, top_k=2, ep_size=2)
    x = workloads.layer_inputs(shape, seed=rank)["x"]
    xs = [torch.empty_like(x) for _ in range(world)]
    dist.all_gather(xs, x)
    out[rank] = (got, bench.job_tokens_per_s(8192, world, got), bool(torch.equal(xs[0], xs[1])))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_report_the_slowest_rank_and_count_all_tokens():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(2, _free_port(), out), nprocs=2, join=True,
                           start_method="spawn")
        res = dict(out)
    for rank in (0, 1):
        ms, tput, same_batch = res[rank]
        assert ms == 5.0
        assert tput == pytest.approx(2 * 8192 / 5e-3)
        assert not same_batch


def _tp_rank_main(rank, world, port, out):
    """TP row split (Hugging Face "Expert parallelism", "With tensor parallelism") as
    real ranks: every rank holds the same batch, dispatches only its slice (the oracle
    layer over its rows, at the rows given by the slice rule), and an all-reduce over
    the group of the zero-padded outputs restores the full output on every rank."""
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import numpy as np
    import oracle
    import workloads
    shape = workloads.LayerShape("tp", N=13, H=16, I=8, E=4, top_k=2, ep_size=2, bias=True)
    inp = workloads.layer_inputs(shape, seed=5)          # the TP group's shared batch
    f64 = {k: (None if v is None else v.double().numpy()) for k, v in inp.items()}
    b, e = oracle.tp_slices(shape.N, world)[rank]
    padded = torch.zeros(shape.N, shape.H, dtype=torch.float64)
    if e > b:
        padded[b:e] = torch.from_numpy(oracle.layer_forward(
            f64["x"][b:e], f64["w_router"], f64["b_router"], f64["w_gate"], f64["w_up"],
            f64["w_down"], shape.top_k, shape.ep_size)["out"])
    dist.all_reduce(padded)
    _, single = oracle.tp_row_split_forward(f64["x"], f64["w_router"], f64["b_router"],
                                            f64["w_gate"], f64["w_up"], f64["w_down"],
                                            shape.top_k, shape.ep_size, world)
    whole = oracle.layer_forward(f64["x"], f64["w_router"], f64["b_router"], f64["w_gate"],
                                 f64["w_up"], f64["w_down"], shape.top_k, shape.ep_size)["out"]
    out[rank] = (float(np.max(np.abs(padded.numpy() - single))),
                 float(np.max(np.abs(padded.numpy() - whole))), e - b)
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_tp_row_split_over_gloo_ranks_restores_the_output(world):
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_tp_rank_main, args=(world, _free_port(), out), nprocs=world,
                           join=True, start_method="spawn")
        res = dict(out)
    sizes = sorted(res[r][2] for r in range(world))
    assert sum(sizes) == 13 and sizes[-1] - sizes[0] <= 1
    for r in range(world):
        to_single, to_whole, _ = res[r]
        assert to_single == 0.0            # the same sum of exact zeros and slice rows
        assert to_whole < 1e-12
