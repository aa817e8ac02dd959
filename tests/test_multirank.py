"""Host logic of the multi-rank paths, on CPU with world_size 2 (gloo).

Batch split (the benchmark): every rank runs its own batch rows (the (b, h) scans share
nothing); the only collectives are the timing barrier and the max over ranks of the
elapsed time.  Rank r's inputs must be rows r*B .. r*B+B-1 of the whole workload.

d_v split (shard.forward_dv_split): every rank scans its column slice with the same
selection and the slices are all-gathered along d_v; here the per-rank scan is the
oracle's on the slice, so the gathered output must equal the oracle's whole-width output
exactly (each column's arithmetic does not depend on the other columns)."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import oracle
from sparse_state_linear_sdm_gb300 import shard
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


def _batch_worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg = wl.B4H8_T2048
        b0, b1 = shard.batch_rows(rank, cfg.B)
        assert b0 == bench.rank_batch_offset(rank, cfg.B)
        out[rank] = wl.inputs(cfg, b0, b1, 0, 2, 0, 8)   # this rank's draw: its rows only
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_each_rank_draws_its_rows_of_the_whole_workload():
    """Rank r's inputs equal rows r*B .. r*B+B-1 of the workload drawn for all ranks at once."""
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_batch_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    cfg = wl.B4H8_T2048
    whole = wl.inputs(cfg, 0, world * cfg.B, 0, 2, 0, 8)
    for r in range(world):
        for k in whole:
            assert np.array_equal(out[r][k], whole[k][r * cfg.B:(r + 1) * cfg.B]), (r, k)


def _dv_problem():
    cfg = wl.TINY_F32
    host = wl.inputs(cfg)
    nh = cfg.B * cfg.H
    kp = host["kp"].reshape(nh, cfg.T, 2, cfg.S)
    qp = host["qp"].reshape(nh, cfg.T, 2, cfg.S)
    v = host["v"].reshape(nh, cfg.T, cfg.d_v)
    a, b = host["alpha"].reshape(nh, cfg.T), host["beta"].reshape(nh, cfg.T)
    M0 = wl.initial_state(cfg, 0, cfg.H)
    return cfg, kp, qp, v, a, b, M0


def _dv_worker(rank, world, port, out):
    import torch
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg, kp, qp, v, a, b, M0 = _dv_problem()
        c0, c1 = shard.dv_columns(cfg.d_v, world, rank)
        iw, sw = oracle.select(kp, cfg.W)                  # the selection, on every rank
        ir, sr = oracle.select(qp, cfg.R)
        M = np.ascontiguousarray(M0[..., c0:c1], dtype=np.float64)
        o_loc = oracle.scan(M, iw, sw, ir, sr, np.ascontiguousarray(v[..., c0:c1]), a, b)
        o = shard.gather_dv(torch.from_numpy(o_loc))
        out[rank] = (c0, c1, o.numpy(), M)
    finally:
        dist.destroy_process_group()


def test_dv_split_gathers_the_whole_output_in_column_order():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_dv_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    cfg, kp, qp, v, a, b, M0 = _dv_problem()
    ref = oracle.forward(kp, qp, v, a, b, M0, cfg.W, cfg.R)
    assert [out[r][:2] for r in range(world)] == [(0, cfg.d_v // 2), (cfg.d_v // 2, cfg.d_v)]
    for r in range(world):
        assert np.array_equal(out[r][2], ref["o"]), f"rank {r}: gathered o differs"
        c0, c1 = out[r][:2]
        assert np.array_equal(out[r][3], ref["M"][..., c0:c1]), f"rank {r}: state slice differs"


def test_dv_columns_partition_d_v():
    for d_v, world in ((128, 1), (128, 2), (128, 4), (128, 8), (64, 2), (16, 4)):
        ranges = [shard.dv_columns(d_v, world, r) for r in range(world)]
        assert ranges[0][0] == 0 and ranges[-1][1] == d_v
        assert all(ranges[i][1] == ranges[i + 1][0] for i in range(world - 1))
        assert all((c1 - c0) % 4 == 0 and c1 > c0 for c0, c1 in ranges)
    with pytest.raises(ValueError):
        shard.dv_columns(24, 4, 0)     # 6 columns per rank: not a multiple of 4
