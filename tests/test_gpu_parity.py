"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Slot indices and scores bit-exact; outputs and final state
within max |x_gpu - x_ref| <= 2e-4 (1 + |x_ref|) (fp32 state vs the fp64 oracle).

Full-size configurations run whole on the GPU in the launch configuration the
benchmark uses; the oracle recomputes a sample of (sequence, head) pairs, each
over its full length (the scan is recurrent, so a head is the unit it can check).
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_state_linear_sdm_gb300 as sdm
from sparse_state_linear_sdm_gb300 import workloads as wl

from sdm_testlib import (TOL, check_against_oracle, device_inputs, device_M0, host_heads, oracle_heads,
                         scaled_err, to_np, torch_dtype)

pytestmark = pytest.mark.gpu

SAMPLED_HEADS = {
    wl.TINY_F32.name: [(0, 0)],
    wl.B4H8_T2048.name: [(0, 0), (1, 3), (2, 5), (3, 7)],
    wl.B8H16_T4096_HOT.name: [(0, 0), (3, 9), (7, 15)],
    wl.B16H4_T8192.name: [(0, 0), (15, 3)],
}
FULL_SIZE = [wl.TINY_F32, wl.B4H8_T2048, wl.B8H16_T4096_HOT, wl.B16H4_T8192]


def _name(cfg):
    return cfg.name


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("cfg", FULL_SIZE, ids=_name)
def test_device_generator_matches_host(cfg):
    T = min(cfg.T, 256)
    d = device_inputs(cfg, T=T)
    for b, h in SAMPLED_HEADS[cfg.name]:
        host = wl.inputs(cfg, b, b + 1, h, h + 1, 0, T)
        for k in ("kp", "qp", "v", "alpha", "beta"):
            assert np.array_equal(to_np(d[k][b, h]), host[k][0, 0]), (cfg.name, k, b, h)
    M0 = device_M0(cfg)
    h, n = cfg.H - 1, min(cfg.N, 4096)
    assert np.array_equal(M0[h, :n].cpu().numpy(), wl.initial_state(cfg, h, h + 1, 0, n)[0])


@pytest.mark.parametrize("cfg", FULL_SIZE, ids=_name)
def test_config_end_to_end(cfg):
    heads = SAMPLED_HEADS[cfg.name]
    d = device_inputs(cfg)
    M0 = device_M0(cfg)
    dev_err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, M, sel = sdm.forward(d["kp"], d["qp"], d["v"], d["alpha"], d["beta"], M0, cfg.W, cfg.R, dev_err=dev_err)
    torch.cuda.synchronize()
    assert dev_err.item() == 0
    del d
    host = host_heads(cfg, heads)
    ref = oracle_heads(cfg, host)
    check_against_oracle(cfg, heads, o, M, sel, ref, label=cfg.name)


def _tie_heavy(rng, shape):
    vals = np.array([-2.0, -1.0, -0.5, -0.0, 0.0, 0.5, 1.0, 1.5, 2.0], np.float32)
    return vals[rng.integers(0, len(vals), size=shape)]


def _rounding_merges(rng, shape, kind):
    """Halves whose fp32 pair sums collapse: one half far larger than the other, so a whole
    row of sums rounds to one value and the flat index alone orders it (which half is the
    large one alternates by token)."""
    n, S = shape[2], shape[4]
    x = np.empty(shape, np.float32)
    for t in range(n):
        if kind == "merge_f32":   # distinct even integers near 2^24 (fp32 spacing 2) + |u| < 1
            big = (2.0 ** 24 + 2.0 * rng.permutation(S)).astype(np.float32)
            small = rng.uniform(-0.9, 0.9, S).astype(np.float32)
        else:                     # Gaussian scores at scales 1e4 and 1e-4
            big = (1e4 * rng.standard_normal(S)).astype(np.float32)
            small = (1e-4 * rng.standard_normal(S)).astype(np.float32)
        x[0, 0, t, t % 2], x[0, 0, t, 1 - t % 2] = big, small
    return x


@pytest.mark.parametrize("S,W,R", [(1, 1, 1), (2, 4, 3), (3, 5, 9), (5, 7, 2), (8, 8, 64), (16, 40, 16),
                                   (17, 33, 5), (32, 8, 8), (64, 100, 64), (100, 128, 1), (256, 32, 200),
                                   (1024, 128, 128), (40, 1024, 512),
                                   (4096, 1024, 7)])   # the library's limits: S = 4096, K = 1024
@pytest.mark.parametrize("kind", ["ties_f32", "gauss_bf16", "gauss_f32", "merge_f32", "scaled_f32"])
def test_select_matches_oracle(S, W, R, kind):
    rng = np.random.default_rng(S * 1000 + W * 7 + R)
    n = 37
    shape = (1, 1, n, 2, S)
    if kind == "ties_f32":
        kp, qp = _tie_heavy(rng, shape), _tie_heavy(rng, shape)
        dt = torch.float32
    elif kind in ("merge_f32", "scaled_f32"):
        kp, qp = _rounding_merges(rng, shape, kind), _rounding_merges(rng, shape, kind)
        dt = torch.float32
    else:
        kp = rng.standard_normal(shape).astype(np.float32)
        qp = rng.standard_normal(shape).astype(np.float32)
        if kind == "gauss_bf16":
            kp, qp = wl.bf16_to_f32(wl.bf16_bits(kp)), wl.bf16_to_f32(wl.bf16_bits(qp))
            dt = torch.bfloat16
        else:
            dt = torch.float32
    kp_d = torch.from_numpy(kp).to("cuda").to(dt)
    qp_d = torch.from_numpy(qp).to("cuda").to(dt)
    iw, sw, ir, sr = sdm.select(kp_d, qp_d, W, R)
    ow, osw = oracle.select(kp[0, 0], W)
    orr, osr = oracle.select(qp[0, 0], R)
    assert np.array_equal(iw[0, 0].cpu().numpy(), ow)
    assert np.array_equal(ir[0, 0].cpu().numpy(), orr)
    assert np.array_equal(sw[0, 0].cpu().numpy(), osw)   # value equality (a zero score may be +0)
    assert np.array_equal(sr[0, 0].cpu().numpy(), osr)


def _random_problem(rng, B, H, T, S, dv, W, R, vdt=torch.float32):
    kp = rng.standard_normal((B, H, T, 2, S)).astype(np.float32)
    qp = rng.standard_normal((B, H, T, 2, S)).astype(np.float32)
    v = rng.standard_normal((B, H, T, dv)).astype(np.float32)
    if vdt == torch.bfloat16:
        v = wl.bf16_to_f32(wl.bf16_bits(v))
    alpha = rng.uniform(0.9, 1.0, (B, H, T)).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, (B, H, T)).astype(np.float32)
    M0 = (0.02 * rng.standard_normal((H, S * S, dv))).astype(np.float32)
    return dict(kp=kp, qp=qp, v=v, alpha=alpha, beta=beta, M0=M0)


def _to_dev(p, vdt=torch.float32):
    d = {k: torch.from_numpy(np.ascontiguousarray(x)).cuda() for k, x in p.items()}
    d["v"] = d["v"].to(vdt)
    return d


def _oracle_problem(p, W, R):
    B, H, T, _, S = p["kp"].shape
    nh = B * H
    M0 = np.broadcast_to(p["M0"][None], (B,) + p["M0"].shape).reshape(nh, S * S, -1)
    return oracle.forward(p["kp"].reshape(nh, T, 2, S), p["qp"].reshape(nh, T, 2, S),
                          p["v"].reshape(nh, T, -1), p["alpha"].reshape(nh, T), p["beta"].reshape(nh, T),
                          M0, W, R)


@pytest.mark.parametrize("B,H,T,S,dv,W,R,vdt", [
    (1, 1, 1, 1, 4, 1, 1, torch.float32),          # N = 1: one slot, every token
    (2, 3, 37, 4, 8, 16, 16, torch.float32),       # W = R = N: every row each token
    (1, 2, 61, 6, 12, 9, 20, torch.bfloat16),      # K > S, ragged sizes
    (2, 2, 300, 8, 32, 5, 3, torch.float32),       # many collisions across tokens
    (1, 1, 200, 16, 64, 64, 64, torch.bfloat16),   # plan chunks span, hash-heavy
    (3, 1, 129, 32, 16, 8, 8, torch.float32),
    (1, 1, 24, 32, 8, 1024, 1024, torch.float32),  # W = R = N = 1024, the slot limit: every row each token
])
def test_scan_edge_cases(B, H, T, S, dv, W, R, vdt):
    rng = np.random.default_rng(B * 100 + T)
    p = _random_problem(rng, B, H, T, S, dv, W, R, vdt)
    d = _to_dev(p, vdt)
    o, M, sel = sdm.forward(d["kp"], d["qp"], d["v"], d["alpha"], d["beta"], d["M0"], W, R)
    ref = _oracle_problem(p, W, R)
    nh = B * H
    assert np.array_equal(sel[0].cpu().numpy().reshape(nh, T, W), ref["idx_w"])
    assert np.array_equal(sel[2].cpu().numpy().reshape(nh, T, R), ref["idx_r"])
    assert scaled_err(o.cpu().numpy().reshape(nh, T, dv), ref["o"]) <= TOL
    assert scaled_err(M.cpu().numpy().reshape(ref["M"].shape), ref["M"]) <= TOL


def test_scan_on_oracle_selection():
    """The scan alone, fed the oracle's own slots and scores."""
    rng = np.random.default_rng(5)
    B, H, T, S, dv, W, R = 2, 2, 150, 16, 32, 12, 10
    p = _random_problem(rng, B, H, T, S, dv, W, R)
    ref = _oracle_problem(p, W, R)
    d = _to_dev(p)
    M = d["M0"][None].repeat(B, 1, 1, 1)
    sel = [torch.from_numpy(ref[k].reshape(B, H, T, -1)).cuda() for k in ("idx_w", "sc_w", "idx_r", "sc_r")]
    o = sdm.scan_forward(M, *sel, d["v"], d["alpha"], d["beta"])
    assert scaled_err(o.cpu().numpy().reshape(B * H, T, dv), ref["o"]) <= TOL
    assert scaled_err(M.cpu().numpy().reshape(ref["M"].shape), ref["M"]) <= TOL


def test_invariants_on_gpu():
    cfg = wl.B4H8_T2048
    d = device_inputs(cfg, T=512)
    M0 = device_M0(cfg)
    # alpha = 1, beta = 0: the state is bit-identical to M0 afterwards
    ones, zeros = torch.ones_like(d["alpha"]), torch.zeros_like(d["beta"])
    o, M, sel = sdm.forward(d["kp"], d["qp"], d["v"], ones, zeros, M0, cfg.W, cfg.R)
    assert torch.equal(M, M0[None].expand_as(M))
    # generic gates: rows never written stay bit-identical to M0
    o, M, sel = sdm.forward(d["kp"], d["qp"], d["v"], d["alpha"], d["beta"], M0, cfg.W, cfg.R)
    for b, h in [(0, 0), (3, 7)]:
        written = torch.zeros(cfg.N, dtype=torch.bool, device="cuda")
        written[sel[0][b, h].flatten().long()] = True
        assert torch.equal(M[b, h][~written], M0[h][~written])
        assert not torch.equal(M[b, h][written], M0[h][written])


def test_chunked_scan_is_bit_identical():
    cfg = wl.B8H16_T4096_HOT   # hot slots: forwarding across the chunk boundary matters
    T = 700
    d = device_inputs(cfg, T=T)
    M0 = device_M0(cfg)
    sel = sdm.select(d["kp"], d["qp"], cfg.W, cfg.R)
    M1 = torch.empty((cfg.B, cfg.H, cfg.N, cfg.d_v), dtype=torch.float32, device="cuda")
    sdm.init_state_from_M0(M1, M0)
    o1 = sdm.scan_forward(M1, *sel, d["v"], d["alpha"], d["beta"])
    M2 = torch.empty_like(M1)
    sdm.init_state_from_M0(M2, M0)
    o2 = torch.empty_like(o1)
    for t0, t1 in [(0, 1), (1, 250), (250, 251), (251, 700)]:
        part = [x[:, :, t0:t1].contiguous() for x in sel]
        o2[:, :, t0:t1] = sdm.scan_forward(M2, *part, d["v"][:, :, t0:t1].contiguous(),
                                           d["alpha"][:, :, t0:t1].contiguous(),
                                           d["beta"][:, :, t0:t1].contiguous())
    assert torch.equal(M1, M2)
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("cfg", [wl.B4H8_T2048, wl.B8H16_T4096_HOT], ids=_name)
def test_forced_shapes_agree(cfg):
    """Every (columns per block, prefetch depth) gives the same state bit for bit
    (the per-row arithmetic does not depend on the shape) and the same outputs up to
    the order of the read reduction."""
    T = 400
    d = device_inputs(cfg, T=T)
    M0 = device_M0(cfg)
    sel = sdm.select(d["kp"], d["qp"], cfg.W, cfg.R)
    results = []
    for cols in (4, 8, 16, 32):
        for pd in (1, 2, 3):
            M = torch.empty((cfg.B, cfg.H, cfg.N, cfg.d_v), dtype=torch.float32, device="cuda")
            sdm.init_state_from_M0(M, M0)
            o = sdm.scan_forward(M, *sel, d["v"], d["alpha"], d["beta"], cols_per_cta=cols, prefetch_depth=pd)
            results.append((cols, pd, o, M))
            if len(results) > 1:
                assert torch.equal(M, results[0][3]), (cols, pd)
                assert scaled_err(o.cpu().numpy(), results[0][2].cpu().numpy()) <= 1e-5, (cols, pd)
                del results[-1]


@pytest.mark.parametrize("dims", [(1, 1, 64, 32, 16, 8, 8), (1, 2, 97, 8, 16, 5, 7), (2, 3, 300, 16, 32, 12, 10)])
def test_workspace_contents_do_not_matter(dims):
    """The planning kernel writes every record field the scan reads: a workspace full of
    garbage gives the same bits as a zeroed one."""
    B, H, T, S, dv, W, R = dims
    rng = np.random.default_rng(sum(dims))
    p = _random_problem(rng, B, H, T, S, dv, W, R, torch.bfloat16)
    d = _to_dev(p, torch.bfloat16)
    sel = sdm.select(d["kp"], d["qp"], W, R)
    results = []
    for fill in (0x00, 0xFF, 0x7F):
        ws = sdm.scan_workspace(B, H, T, dv, W, R, "cuda")
        ws.fill_(fill)
        M = d["M0"][None].repeat(B, 1, 1, 1)
        o = sdm.scan_forward(M, *sel, d["v"], d["alpha"], d["beta"], workspace=ws)
        results.append((o, M))
    for o, M in results[1:]:
        assert torch.equal(o, results[0][0]) and torch.equal(M, results[0][1])


def test_device_error_flags():
    rng = np.random.default_rng(9)
    B, H, T, S, dv, W, R = 1, 1, 20, 8, 8, 4, 4
    p = _random_problem(rng, B, H, T, S, dv, W, R)
    d = _to_dev(p)
    M = d["M0"][None].contiguous()
    iw, sw, ir, sr = sdm.select(d["kp"], d["qp"], W, R)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = iw.clone()
    bad[0, 0, 5, 1] = S * S + 7          # out of range
    bad[0, 0, 9, 2] = -3
    sdm.scan_forward(M.clone(), bad, sw, ir, sr, d["v"], d["alpha"], d["beta"], dev_err=err)
    assert err.item() & sdm.SDM_DEV_INDEX_RANGE
    err.zero_()
    dup = iw.clone()
    dup[0, 0, 4, 3] = dup[0, 0, 4, 0]
    sdm.scan_forward(M.clone(), dup, sw, ir, sr, d["v"], d["alpha"], d["beta"], dev_err=err)
    assert err.item() & sdm.SDM_DEV_DUP_WRITE
    err.zero_()
    sdm.scan_forward(M.clone(), iw, sw, ir, sr, d["v"], d["alpha"], d["beta"], dev_err=err)
    torch.cuda.synchronize()
    assert err.item() == 0


def test_empty_sequence_is_a_no_op():
    M = torch.randn(1, 1, 16, 8, device="cuda")
    before = M.clone()
    e = torch.empty(1, 1, 0, 4, dtype=torch.int32, device="cuda")
    s = torch.empty(1, 1, 0, 4, dtype=torch.float32, device="cuda")
    o = sdm.scan_forward(M, e, s, e, s, torch.empty(1, 1, 0, 8, device="cuda"),
                         torch.empty(1, 1, 0, device="cuda"), torch.empty(1, 1, 0, device="cuda"))
    assert o.shape == (1, 1, 0, 8) and torch.equal(M, before)


def test_overlapped_forward_waits_for_earlier_work_on_the_state():
    """forward(overlap=True) initialises M on a side stream: that stream must first wait for
    work already queued on the caller's stream.  A delayed copy of M queued there must
    still see the finished state, not the next call's initialisation."""
    cfg = wl.B4H8_T2048
    d = device_inputs(cfg)
    M0 = device_M0(cfg)
    _, ref, _ = sdm.forward(d["kp"], d["qp"], d["v"], d["alpha"], d["beta"], M0, cfg.W, cfg.R, overlap=False)
    torch.cuda.synchronize()
    M = torch.empty_like(ref)
    sdm.forward(d["kp"], d["qp"], d["v"], d["alpha"], d["beta"], M0, cfg.W, cfg.R, M=M)
    torch.cuda._sleep(50_000_000)  # keeps the caller's stream busy for tens of milliseconds
    snap = M.clone()
    sdm.forward(d["kp"], d["qp"], d["v"], d["alpha"], d["beta"], M0, cfg.W, cfg.R, M=M)
    torch.cuda.synchronize()
    assert torch.equal(snap, ref)
    assert torch.equal(M, ref)
