"""The pipelined forward (sdm_forward): selection of token chunk c+1 and planning overlap
the scan of chunk c on the library's own streams.  A chunk boundary is a fresh scan
pipeline, exactly like chained sdm_scan_forward calls, so every result must equal the
one-stream path (initialisation, selection, scan) bit for bit, for any chunking."""
import numpy as np
import pytest
import torch

import sparse_state_linear_sdm_gb300 as sdm
from sparse_state_linear_sdm_gb300 import workloads as wl

from sdm_testlib import TOL, device_inputs, device_M0, scaled_err

pytestmark = pytest.mark.gpu


def _run(d, M0, W, R, **kw):
    o, M, sel = sdm.forward(d["kp"], d["qp"], d["v"], d["alpha"], d["beta"], M0, W, R, **kw)
    torch.cuda.synchronize()
    return o, M, sel


def _assert_same(a, b, label):
    o1, M1, s1 = a
    o2, M2, s2 = b
    for x, y, name in zip(s1, s2, ("idx_w", "sc_w", "idx_r", "sc_r")):
        assert torch.equal(x, y), (label, name)
    assert torch.equal(M1, M2), (label, "M")
    assert torch.equal(o1, o2), (label, "o")


@pytest.mark.parametrize("cfg", [wl.B4H8_T2048, wl.B8H16_T4096_HOT], ids=lambda c: c.name)
def test_pipelined_forward_equals_one_stream_path(cfg):
    d = device_inputs(cfg)
    M0 = device_M0(cfg)
    ref = _run(d, M0, cfg.W, cfg.R, overlap=False)
    for chunks in (0, 1, 3, 7):
        _assert_same(_run(d, M0, cfg.W, cfg.R, chunks=chunks), ref, (cfg.name, chunks))


def _random(rng, B, H, T, S, dv, dt):
    kp = torch.from_numpy(rng.standard_normal((B, H, T, 2, S)).astype(np.float32)).cuda().to(dt)
    qp = torch.from_numpy(rng.standard_normal((B, H, T, 2, S)).astype(np.float32)).cuda().to(dt)
    v = torch.from_numpy(rng.standard_normal((B, H, T, dv)).astype(np.float32)).cuda().to(dt)
    alpha = torch.from_numpy(rng.uniform(0.9, 1.0, (B, H, T)).astype(np.float32)).cuda()
    beta = torch.from_numpy(rng.uniform(0.0, 1.0, (B, H, T)).astype(np.float32)).cuda()
    M0 = torch.from_numpy((0.02 * rng.standard_normal((H, S * S, dv))).astype(np.float32)).cuda()
    return dict(kp=kp, qp=qp, v=v, alpha=alpha, beta=beta), M0


@pytest.mark.parametrize("B,H,T,S,dv,W,R,dt,chunks", [
    (1, 1, 1, 4, 8, 3, 2, torch.float32, 0),       # one token
    (1, 2, 5, 6, 12, 9, 20, torch.bfloat16, 8),    # more chunks asked than tokens; K > S
    (2, 3, 37, 8, 16, 16, 16, torch.float32, 4),   # ragged last chunk; W = R = N / 4
    (2, 1, 300, 16, 64, 64, 64, torch.bfloat16, 7),  # rows forwarded across many tokens
    (1, 1, 2500, 32, 32, 8, 8, torch.float32, 0),  # automatic chunking: 3 chunks, ragged
])
def test_pipelined_forward_ragged_and_small(B, H, T, S, dv, W, R, dt, chunks):
    rng = np.random.default_rng(B * 7 + H * 11 + T + S)
    d, M0 = _random(rng, B, H, T, S, dv, dt)
    ref = _run(d, M0, W, R, overlap=False)
    _assert_same(_run(d, M0, W, R, chunks=chunks), ref, (B, H, T, chunks))


def test_pipelined_forward_continues_from_the_state_in_M():
    """M0=None continues from M: two calls over T1 and T2 tokens equal one call over both."""
    cfg = wl.B4H8_T2048
    d = device_inputs(cfg)
    M0 = device_M0(cfg)
    o_all, M_all, _ = _run(d, M0, cfg.W, cfg.R, chunks=3)
    T1 = 700
    part = lambda t0, t1: {k: x[:, :, t0:t1].contiguous() for k, x in d.items()}
    o1, M, _ = _run(part(0, T1), M0, cfg.W, cfg.R, chunks=2)
    o2, M, _ = _run(part(T1, cfg.T), None, cfg.W, cfg.R, M=M, chunks=2)
    assert torch.equal(M, M_all)
    assert torch.equal(torch.cat([o1, o2], dim=2), o_all)


def test_pipelined_forward_scan_events_bracket_each_scan_kernel():
    cfg = wl.B4H8_T2048
    d = device_inputs(cfg)
    M0 = device_M0(cfg)
    n = sdm.forward_chunks(cfg.T, 4)
    assert n == 4
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n)]
    _run(d, M0, cfg.W, cfg.R, chunks=4, scan_events=evs)
    times = [evs[2 * c].elapsed_time(evs[2 * c + 1]) for c in range(n)]
    assert all(t > 0 for t in times)
    # the chunks' scans run one after the other
    assert all(evs[2 * c + 1].elapsed_time(evs[2 * c + 2]) >= 0 for c in range(n - 1))


def test_pipelined_forward_matches_the_oracle_on_a_small_case():
    import oracle
    rng = np.random.default_rng(5)
    B, H, T, S, dv, W, R = 1, 2, 40, 8, 16, 6, 5
    d, M0 = _random(rng, B, H, T, S, dv, torch.float32)
    o, M, sel = _run(d, M0, W, R, chunks=3)
    host = {k: x.cpu().numpy() for k, x in d.items()}
    nh = B * H
    ref = oracle.forward(host["kp"].reshape(nh, T, 2, S), host["qp"].reshape(nh, T, 2, S),
                         host["v"].reshape(nh, T, dv), host["alpha"].reshape(nh, T),
                         host["beta"].reshape(nh, T), np.broadcast_to(M0.cpu().numpy()[None], (B, H, S * S, dv))
                         .reshape(nh, S * S, dv), W, R)
    assert np.array_equal(sel[0].cpu().numpy().reshape(nh, T, W), ref["idx_w"])
    assert np.array_equal(sel[2].cpu().numpy().reshape(nh, T, R), ref["idx_r"])
    assert scaled_err(o.cpu().numpy().reshape(nh, T, dv), ref["o"]) <= TOL
    assert scaled_err(M.cpu().numpy().reshape(nh, S * S, dv), ref["M"]) <= TOL


@pytest.mark.parametrize("B,H,T,S,dv,W,R,chunks", [
    (2, 2, 1, 32, 16, 2, 8, 0),       # one token: almost every row keeps M_0
    (1, 3, 3, 32, 8, 2, 16, 2),       # rows read before any token writes them
    (2, 1, 50, 8, 16, 4, 16, 3),      # N = 64: rows written, read, rewritten across chunks
    (1, 2, 257, 16, 32, 32, 32, 5),   # most rows written somewhere, ragged last chunk
])
def test_pipelined_forward_from_M0_writes_every_row(B, H, T, S, dv, W, R, chunks):
    """M starts as NaN and the workspace as garbage: every row of the result must come from
    M_0 or from the scan, exactly as on the one-stream path."""
    rng = np.random.default_rng(T * 13 + S)
    d, M0 = _random(rng, B, H, T, S, dv, torch.float32)
    ref = _run(d, M0, W, R, overlap=False)
    M = torch.full((B, H, S * S, dv), float("nan"), device="cuda")
    ws = sdm.forward_workspace(B, H, T, dv, W, R, "cuda", chunks)
    ws.copy_(torch.randint(0, 256, ws.shape, dtype=torch.uint8, device="cuda"))
    got = _run(d, M0, W, R, chunks=chunks, M=M, workspace=ws)
    _assert_same(got, ref, (B, H, T, S, chunks))


NAMES = ("kp", "qp", "v", "alpha", "beta")


def test_copy_token_window_moves_exactly_its_tokens():
    cfg = wl.B4H8_T2048
    d = device_inputs(cfg, T=100)
    host = {k: d[k].cpu().pin_memory() for k in NAMES}
    for k in NAMES:
        dst = torch.full_like(d[k], -7.0)
        sdm.copy_token_window(dst, host[k], 30, 77)       # host -> device
        sdm.copy_token_window(dst, d[k], 0, 5)            # device -> device
        torch.cuda.synchronize()
        assert torch.equal(dst[:, :, 30:77], d[k][:, :, 30:77]), k
        assert torch.equal(dst[:, :, 0:5], d[k][:, :, 0:5]), k
        assert bool((dst[:, :, 5:30] == -7.0).all()) and bool((dst[:, :, 77:] == -7.0).all()), k
        back = torch.zeros_like(host[k]).pin_memory()
        sdm.copy_token_window(back, dst, 30, 77)          # device -> host
        torch.cuda.synchronize()
        assert torch.equal(back[:, :, 30:77], host[k][:, :, 30:77]), k


def test_pinned_empty_is_page_locked_and_round_trips():
    x = torch.randn(3, 5, 77, 9, device="cuda")
    h = sdm.pinned_empty(x.shape, x.dtype)
    assert h.is_pinned() and h.shape == x.shape and h.dtype == x.dtype
    h.copy_(x, non_blocking=True)
    y = torch.empty_like(x)
    y.copy_(h, non_blocking=True)
    torch.cuda.synchronize()
    assert torch.equal(y, x)
    b = sdm.pinned_empty((4, 2, 10, 2, 8), torch.bfloat16)
    assert b.is_pinned() and b.dtype == torch.bfloat16
    del h, b  # the registration goes with the buffers


def test_pinned_empty_large_buffer_on_huge_page_boundary():
    """A buffer of at least a quarter of the host's huge page takes the huge-page path: it
    starts on a huge-page boundary, is page-locked and round-trips through the GPU."""
    from sparse_state_linear_sdm_gb300 import api
    huge = api._huge_page_bytes()
    n = (huge // 4 + (1 << 20)) // 4
    h = sdm.pinned_empty((n,), torch.float32)
    assert h.is_pinned() and h.numel() == n
    assert h.data_ptr() % huge == 0
    x = torch.arange(n, dtype=torch.float32, device="cuda")
    h.copy_(x, non_blocking=True)
    y = torch.empty_like(x)
    y.copy_(h, non_blocking=True)
    torch.cuda.synchronize()
    assert torch.equal(y, x)
    del h


@pytest.mark.parametrize("chunks", [3, 4])
def test_inputs_arriving_window_by_window(chunks):
    """The batch's inputs copied from pinned host memory one token window at a time on a
    copy stream, the pass waiting for each window's copy before its chunk's selection
    (sdm_forward_streamed): the same bits as with the inputs resident."""
    cfg = wl.B4H8_T2048
    d = device_inputs(cfg)
    M0 = device_M0(cfg)
    ref = _run(d, M0, cfg.W, cfg.R, chunks=chunks)
    host = {k: sdm.pinned_empty(d[k].shape, d[k].dtype) for k in NAMES}
    for k in NAMES:
        host[k].copy_(d[k])
    dst = {k: torch.full_like(d[k], float("nan")) for k in NAMES}
    torch.cuda.synchronize()
    n = sdm.forward_chunks(cfg.T, chunks)
    Tc = -(-cfg.T // n)
    copy = torch.cuda.Stream()
    evs = []
    for c in range(n):
        for k in NAMES:
            sdm.copy_token_window(dst[k], host[k], c * Tc, min(cfg.T, (c + 1) * Tc), stream=copy)
        e = torch.cuda.Event()
        e.record(copy)
        evs.append(e)
    got = _run(dst, M0, cfg.W, cfg.R, chunks=chunks, input_events=evs)
    _assert_same(got, ref, ("window by window", chunks))

