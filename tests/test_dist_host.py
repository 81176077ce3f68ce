"""The bench's multi-rank host logic on CPU: two gloo ranks, each with its
own problem (distinct seeds, no data exchange), the step time reduced with
MAX over ranks, and the whole-job throughput counting every rank's work."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        return sk.getsockname()[1]


def _rank_main(rank, ws, port, queue):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import bench
        from hierarchical_sparse_attention_mean_gb300 import synth
        w = bench.rank_workload(synth.WORKLOADS[synth.HEADLINE], rank)
        small = synth.Workload(**{**w.__dict__, "n": 1024, "heads": 1, "kind": "iid", "grid": (32, 32)})
        x = synth.make_inputs(small, with_dout=False, threads=1)
        t_local = 10.0 + 5.0 * rank                    # rank 1 is the slower one
        t_max = bench.max_over_ranks(t_local, ws, torch.device("cpu"))
        dist.barrier()
        queue.put((rank, w.seed, float(x["q"][0, 0, 0]), t_max))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_independent_problems_max_time():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, queue)) for r in range(ws)]
    for p in procs:
        p.start()
    res = sorted(queue.get(timeout=240) for _ in range(ws))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, seed0, v0, t0), (r1, seed1, v1, t1) = res
    assert seed0 != seed1 and v0 != v1            # each rank draws its own inputs
    assert t0 == t1 == 15.0                        # both ranks see the slowest rank's time


def test_job_value_counts_every_rank():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_value(1, 92.3e9, 1.6)
    two = bench.job_value(2, 92.3e9, 1.6)
    assert abs(two - 2 * one) < 1e-9 and abs(one - 92.3e9 / 1.6e-3 / 1e12) < 1e-9
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
