"""The multi-GPU path is replicas only (one process per GPU, each running the whole
prefill on its own seeded inputs, no data exchange): this covers its host logic on the
CPU with two gloo ranks, with the same functions bench.py uses under torchrun. Each
rank's timings become the maximum over the ranks, and the job's throughput is the
tokens of all ranks over that time."""
import os
import socket
import sys
from pathlib import Path

import torch
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parents[1]


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, str(ROOT))
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workloads as W
        # rank-dependent timings: rank r took 1 + r ms for the prefill and 5 - r for the step
        times = bench.max_over_ranks([1.0 + rank, 5.0 - rank], world, torch.device("cpu"))
        value = bench.job_throughput(world, 65536, times[0])
        # each replica draws its own inputs (seed 4 + rank), as bench.py does
        wl = W.long_prefill(seed=4 + rank, tokens=64, decode_steps=1)
        q.put((rank, times, value, float(wl.xBC[:4].float().sum())))
        torch.distributed.barrier()
    finally:
        torch.distributed.destroy_process_group()


def test_replica_timing_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    try:
        got = sorted(q.get(timeout=120) for _ in range(world))
    finally:
        for pr in procs:
            pr.join(timeout=60)
            if pr.is_alive():
                pr.kill()
    assert [pr.exitcode for pr in procs] == [0, 0]
    for rank, times, value, _ in got:
        assert times == [2.0, 5.0], (rank, times)  # max over ranks of (1, 2) and (5, 4)
        assert value == world * 65536 / 2.0e-3
    assert got[0][3] != got[1][3], "replicas must draw different inputs"


def test_single_rank_is_identity():
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench.max_over_ranks([3.0, 4.0], 1, torch.device("cpu")) == [3.0, 4.0]
    assert bench.job_throughput(1, 65536, 1.0) == 65536 / 1e-3
