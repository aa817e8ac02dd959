"""Host logic of the multi-rank benchmark path, on CPU with world_size 2 (gloo).

Every rank runs its own batch rows (the (b, h) scans share nothing); the only
collectives are the timing barrier and the max over ranks of the elapsed time."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from sparse_state_linear_sdm_gb300 import workloads as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env()[:2] == (rank, world)
        ms = 10.0 + 7.0 * rank                     # rank 1 is the slow one
        m = bench.max_over_ranks(ms, "cpu")
        cfg = wl.B4H8_T2048
        b0 = bench.rank_batch_offset(rank, cfg.B)
        kp = wl.halves(cfg, wl.FIELD_KP, b0, b0 + 1, 0, 1, 0, 4)
        out[rank] = (m, b0, float(kp.sum()))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_ranks_share_max_time_and_disjoint_batches():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    (m0, b00, s0), (m1, b01, s1) = out[0], out[1]
    assert m0 == m1 == 17.0
    assert (b00, b01) == (0, wl.B4H8_T2048.B)
    assert s0 != s1                                  # different sequences per rank
    # whole-job throughput: both ranks' units over the slowest rank's time
    assert bench.whole_job_rate(1000, 5, world, 17.0) == pytest.approx(2 * 1000 * 5 / 0.017)


def test_single_process_max_is_identity():
    assert bench.max_over_ranks(3.5, "cpu") == 3.5
