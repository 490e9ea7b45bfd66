"""The N>1 path of the benchmark: one replica per rank, no collective on the
data path, whole-job throughput = all ranks' steps / the slowest rank's time.
Runs as two gloo ranks on the CPU (each rank also runs the oracle on its own
replica batch, so the per-rank work is real and independent)."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    from top_sparse_attention_pks_gb300.workloads import WORKLOADS, draw_host
    # each rank serves its own replica batch (seed offset = rank): top-k on
    # its own scores, no exchange between ranks
    wl = WORKLOADS["paging_example"]
    h = draw_host(wl)
    rng = np.random.default_rng(100 + rank)
    lens = h["seq_lens"].numpy()
    scores = rng.integers(-1000, 1000, size=(wl.B, int(lens.max())), dtype=np.int64)
    idx = oracle.topk(lens, scores, wl.k)
    # rank r pretends its 3 steps took (r + 1) seconds
    value, total = bench.job_throughput(rank + 1.0, 3, world, dist)
    out[rank] = (value, total, int((idx >= 0).sum()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn")
    lens_sel = min(403, 64) + min(96, 64) + min(241, 64) + min(30, 64) + min(176, 64)
    for r in range(world):
        value, total, n_sel = out[r]
        assert total == pytest.approx(2.0)          # max over ranks
        assert value == pytest.approx(2 * 3 / 2.0)  # all ranks' steps / slowest time
        assert n_sel == lens_sel                     # each replica's own selection


def test_single_rank_needs_no_process_group():
    import bench
    value, total = bench.job_throughput(0.5, 10, 1, None)
    assert (value, total) == (20.0, 0.5)
