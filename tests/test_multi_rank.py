"""The multi-rank (N > 1) host logic of bench.py on CPU: two gloo ranks,
each with its own query batches (no collective on the data), the timing
reduced to the slowest rank, and the whole-job rate from it."""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    import qsa_inputs as qi
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        n = 8
        variants = list(bench.rank_variants(rank, n))
        w = qi.WORKLOADS[0]
        q0, _ = qi.make_inputs(w, variant=variants[0])
        local_ms = 10.0 + 5.0 * rank                      # rank 1 is the slower one
        t_max = bench.max_over_ranks(torch, dist, local_ms, torch.device("cpu"))
        rate = bench.aggregate_rate(world, bench.units_per_step(w) * 4, t_max)
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), variants=np.array(variants), q0=q0,
                 t_max=t_max, rate=rate)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    torch.multiprocessing.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                                join=True)
    r = [np.load(tmp_path / f"rank{i}.npz") for i in range(world)]
    # distinct input sets per rank, together covering world x n variants
    v0, v1 = set(r[0]["variants"].tolist()), set(r[1]["variants"].tolist())
    assert not (v0 & v1) and len(v0 | v1) == 16
    assert not np.array_equal(r[0]["q0"], r[1]["q0"])
    # every rank sees the slowest rank's time, and the same whole-job rate
    assert float(r[0]["t_max"]) == float(r[1]["t_max"]) == 15.0
    sys.path.insert(0, ROOT)
    import bench
    import qsa_inputs as qi
    want = world * bench.units_per_step(qi.WORKLOADS[0]) * 4 / 0.015
    assert float(r[0]["rate"]) == pytest.approx(want) and float(r[1]["rate"]) == pytest.approx(want)
