"""Projections x -> k', q' on the tensor cores (sdm_project_kq through the C ABI) against
the oracle's fp64 projection, then the selection on the projected halves against the
oracle's selection on the same halves.

Tolerance, per output: the kernel rounds an fp32 accumulation of exact bf16 products to
bf16, so  |g - r| <= 2^-8 |r| + 4 D 2^-24 sum_d |x_d w_nd|  (half a bf16 unit of the
result, plus four times the worst-case error of D fp32 additions in any order); in
addition at least 95 % of the outputs must equal the correctly rounded sum.  A wrong
index, a dropped K block or a transposed operand gives errors of the order of the
values themselves."""
import numpy as np
import pytest
import torch

import oracle
import sparse_state_linear_sdm_gb300 as sdm
from sparse_state_linear_sdm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _f32(t):
    return t.float().cpu().numpy()


def _inputs(seed, B, T, D, H, S):
    xb = wl.projection_features(seed, B, T, D).reshape(B, T, D)
    wb = wl.projection_weights(seed, H, S, D)
    return xb, wb


def _check(got, want, mag, D, label):
    got = np.asarray(got, np.float64)
    tol = 2.0 ** -8 * np.abs(want) + 4 * D * 2.0 ** -24 * mag
    err = np.abs(got - want)
    bad = err > tol
    assert not bad.any(), f"{label}: {bad.sum()} outputs out of bound, worst {float((err - tol).max()):.3e}"
    rn = wl.bf16_to_f32(wl.bf16_bits(want.astype(np.float32)))
    frac = float(np.mean(got == rn)) if got.size else 1.0
    assert frac >= 0.95, f"{label}: only {frac:.3f} of outputs correctly rounded"


def _run(xb, wb, H, S, max_ctas=0, pair=-1):
    x, w = _bf16_dev(xb), _bf16_dev(wb)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kp, qp = sdm.project_kq(x, w, H, S, dev_err=err, max_ctas=max_ctas, pair=pair)
    torch.cuda.synchronize()
    assert err.item() == 0
    return kp, qp


@pytest.mark.parametrize("pair", [0, 2])
@pytest.mark.parametrize("B,T,D,H,S,max_ctas", [
    (1, 1, 8, 1, 4, 0),          # one token, D < one K block, 16 output columns
    (2, 100, 72, 2, 6, 0),       # 2S % 8 != 0 (column-wise stores), ragged K block
    (1, 300, 128, 1, 64, 0),     # one column tile, ragged (and, paired, empty) row tiles
    (2, 257, 512, 4, 128, 0),    # 5 x 8 tiles
    (2, 257, 512, 4, 128, 4),    # the same on 4 blocks: ~10-20 tiles each, accumulators alternate
    (1, 70, 256, 2, 64, 2),      # one block (or one pair) runs every tile
    (9, 300, 64, 1, 128, 0),     # several groups of row tiles in the tile order
    (1, 129, 2048, 4, 1024, 0),  # the full-size output width and depth, two row tiles
])
def test_projection_matches_oracle(B, T, D, H, S, max_ctas, pair):
    xb, wb = _inputs(B * 31 + T + D, B, T, D, H, S)
    kp, qp = _run(xb, wb, H, S, max_ctas, pair)
    rk, rq, (mk, mq) = oracle.project(wl.bf16_to_f32(xb), wl.bf16_to_f32(wb), H, S)
    _check(_f32(kp), rk, mk, D, ("kp", B, T, D, H, S, max_ctas, pair))
    _check(_f32(qp), rq, mq, D, ("qp", B, T, D, H, S, max_ctas, pair))


def test_block_counts_agree_bit_for_bit():
    """Every block count accumulates each output in the same order (K blocks in sequence,
    the same MMA shape), so the results are identical; the same for the 2-SM shape."""
    B, T, D, H, S = 3, 200, 320, 2, 128
    xb, wb = _inputs(99, B, T, D, H, S)
    k1, q1 = _run(xb, wb, H, S, 0, 0)
    k2, q2 = _run(xb, wb, H, S, 5, 0)
    k3, q3 = _run(xb, wb, H, S, 0, 2)
    k4, q4 = _run(xb, wb, H, S, 6, 2)
    assert torch.equal(k1, k2) and torch.equal(q1, q2)
    assert torch.equal(k3, k4) and torch.equal(q3, q4)


def test_two_sm_tiles_on_few_pairs():
    """The 2-SM shape (tcgen05 cta_group::2) with one and three pairs: each pair runs many
    256 x 256 tiles, so both accumulators and every stage wrap many times."""
    B, T, D, H, S = 2, 300, 384, 2, 128
    xb, wb = _inputs(123, B, T, D, H, S)
    rk, rq, (mk, mq) = oracle.project(wl.bf16_to_f32(xb), wl.bf16_to_f32(wb), H, S)
    for ctas in (2, 6):
        kp, qp = _run(xb, wb, H, S, ctas, 2)
        _check(_f32(kp), rk, mk, D, ("kp 2sm", ctas))
        _check(_f32(qp), rq, mq, D, ("qp 2sm", ctas))


def test_projected_halves_select_like_the_oracle():
    """Selection on the projected bf16 halves: the GPU's slots and scores equal the oracle's
    selection run on the same halves (the decision is taken on identical values)."""
    B, T, D, H, S, W, R = 2, 64, 256, 2, 64, 32, 24
    xb, wb = _inputs(7, B, T, D, H, S)
    kp, qp = _run(xb, wb, H, S)
    iw, sw, ir, sr = sdm.select(kp, qp, W, R)
    torch.cuda.synchronize()
    hk = _f32(kp).reshape(B * H, T, 2, S)
    hq = _f32(qp).reshape(B * H, T, 2, S)
    oiw, osw = oracle.select(hk, W)
    oir, osr = oracle.select(hq, R)
    assert np.array_equal(iw.cpu().numpy().reshape(oiw.shape), oiw)
    assert np.array_equal(ir.cpu().numpy().reshape(oir.shape), oir)
    assert np.array_equal(sw.cpu().numpy().reshape(osw.shape), osw)
    assert np.array_equal(sr.cpu().numpy().reshape(osr.shape), osr)


def test_projection_full_workload_sampled_tokens():
    """B16 T8192 D2048 H4 S1024 (every k', q' of the default selection workload) in the
    launch configuration the benchmark times; the oracle on 48 sampled tokens."""
    B, T, D, H, S = 16, 8192, wl.PROJ_D, 4, 1024
    seed = 3
    xb = wl.projection_features(seed, B, T, D)
    wb = wl.projection_weights(seed, H, S, D)
    x = _bf16_dev(xb).view(B, T, D)
    kp, qp = _run_dev(x, _bf16_dev(wb), H, S)
    rng = np.random.default_rng(5)
    ms = np.sort(rng.choice(B * T, 48, replace=False))
    ms[0], ms[-1] = 0, B * T - 1
    rk, rq, (mk, mq) = oracle.project(wl.bf16_to_f32(xb[ms]), wl.bf16_to_f32(wb), H, S)  # [48, H, 2, S]
    b, t = ms // T, ms % T
    bi, ti = torch.from_numpy(b).cuda(), torch.from_numpy(t).cuda()
    gk = _f32(kp[bi, :, ti])   # [48, H, 2, S]
    gq = _f32(qp[bi, :, ti])
    _check(gk, rk, mk, D, "kp sampled")
    _check(gq, rq, mq, D, "qp sampled")


def _run_dev(x, w, H, S):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kp, qp = sdm.project_kq(x, w, H, S, dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    return kp, qp


def test_projection_rejects_bad_arguments():
    x = torch.zeros((1, 4, 12), dtype=torch.bfloat16, device="cuda")   # D % 8 != 0
    w = torch.zeros((4 * 1 * 4, 12), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(sdm.SDMError):
        sdm.project_kq(x, w, 1, 4)


def test_bounded_wait_runs_out_and_reports_a_timeout():
    """The projection kernel's mbarrier wait, on a phase that nothing completes, gives up
    after its limit and reports SDM_DEV_TIMEOUT; on a completed phase it returns at once
    without an error; with the block's stop flag already raised it gives up at once.  The
    context stays usable: a projection afterwards is still correct."""
    limit = 1_000_000                                        # 1 ms
    err, ns = sdm.bounded_wait_check(0, limit)
    assert err == sdm.SDM_DEV_TIMEOUT
    assert limit <= ns < limit + 200_000_000, ns
    err, ns = sdm.bounded_wait_check(1, limit)
    assert err == 0 and ns < limit, (err, ns)
    err, ns = sdm.bounded_wait_check(2, 500_000_000)         # left by the flag, not the timer
    assert err == sdm.SDM_DEV_TIMEOUT and ns < 100_000_000, (err, ns)
    B, T, D, H, S = 1, 64, 64, 1, 32
    xb, wb = _inputs(5, B, T, D, H, S)
    kp, qp = _run(xb, wb, H, S)
    rk, rq, (mk, mq) = oracle.project(wl.bf16_to_f32(xb), wl.bf16_to_f32(wb), H, S)
    _check(_f32(kp), rk, mk, D, "kp after the timeouts")
    _check(_f32(qp), rq, mq, D, "qp after the timeouts")


@pytest.mark.parametrize("pair,cta,step", [
    (0, 0, 3),    # single blocks: the MMAs wait for a copy that is never issued
    (2, 1, 0),    # pairs: the peer never issues; the leader's phases miss the peer's half
    (2, 1, 9),    # ... after 9 K steps: the leader runs up to a round of stages ahead
    (2, 0, 3),    # the leader stops issuing; the peer issues phases the leader never armed
    (2, 0, 9),
])
def test_stalled_producer_stops_drains_and_reports(pair, cta, step):
    """A producer that stops issuing copies part-way (sdm_test_project_stall, 1 ms wait
    limit): the waits for its copies run out, the blocks stop, drain every copy in flight
    (in a pair, the phases only one block issued too) and report SDM_DEV_TIMEOUT, well
    inside the 2 s limit of a drain wait that never completes.  A projection afterwards is
    still correct."""
    import time
    B, T, D, H, S = 2, 300, 1024, 2, 128      # 16 K steps per tile
    xb, wb = _inputs(77, B, T, D, H, S)
    x, w = _bf16_dev(xb).view(B, T, D), _bf16_dev(wb)
    t0 = time.perf_counter()
    err = sdm.project_stall_check(x, w, H, S, pair, cta, step, 1_000_000)
    elapsed = time.perf_counter() - t0
    assert err & sdm.SDM_DEV_TIMEOUT, err
    assert elapsed < 1.5, elapsed
    kp, qp = _run(xb, wb, H, S, 0, pair)
    rk, rq, (mk, mq) = oracle.project(wl.bf16_to_f32(xb), wl.bf16_to_f32(wb), H, S)
    _check(_f32(kp), rk, mk, D, ("kp after a stall", pair, cta, step))
    _check(_f32(qp), rq, mq, D, ("qp after a stall", pair, cta, step))
