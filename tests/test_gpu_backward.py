"""Backward pass on the GPU (sdm_scan_forward_train + sdm_scan_backward +
sdm_select_backward, through the C ABI) against the oracle's pinned backward, on the
GPU's own selection.

Tolerance, per gradient tensor (normwise): max |g - r| <= 2e-4 * (1 + max |r|).  The score
gradients come out of a cancelling difference (softmax backward: dk - <k, dk>), so an
elementwise relative bound would measure the cancellation, not the kernel; 2e-4 is the
forward's fp32 bound, taken at the scale of each gradient."""
import numpy as np
import pytest
import torch

import oracle
import sparse_state_linear_sdm_gb300 as sdm
from sparse_state_linear_sdm_gb300 import workloads as wl

from sdm_testlib import device_inputs, device_M0, to_np

pytestmark = pytest.mark.gpu
GTOL = 2e-4


def normwise(got, want) -> float:
    g = np.asarray(got, np.float64)
    w = np.asarray(want, np.float64)
    assert g.shape == w.shape, (g.shape, w.shape)
    return float(np.abs(g - w).max() / (1.0 + np.abs(w).max())) if g.size else 0.0


def _random(rng, B, H, T, S, dv, vdt):
    f = lambda *sh: rng.standard_normal(sh).astype(np.float32)
    d = dict(kp=f(B, H, T, 2, S), qp=f(B, H, T, 2, S), v=f(B, H, T, dv),
             alpha=rng.uniform(0.85, 1.0, (B, H, T)).astype(np.float32),
             beta=rng.uniform(0.1, 1.0, (B, H, T)).astype(np.float32))
    if vdt == torch.bfloat16:
        d["v"] = wl.bf16_to_f32(wl.bf16_bits(d["v"]))
    dev = {k: torch.from_numpy(x).cuda() for k, x in d.items()}
    dev["v"] = dev["v"].to(vdt)
    M0 = (0.3 * rng.standard_normal((H, S * S, dv))).astype(np.float32)
    dO = f(B, H, T, dv)
    dMT = f(B, H, S * S, dv)
    return d, dev, M0, dO, dMT


def _gpu_backward(dev, M0, dO, dMT, W, R):
    B, H, T, _, S = dev["kp"].shape
    dv = dev["v"].shape[-1]
    sel = sdm.select(dev["kp"], dev["qp"], W, R)
    M = torch.from_numpy(np.broadcast_to(M0[None], (B,) + M0.shape).copy()).cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, w_prev, r_rows = sdm.scan_forward_train(M, *sel, dev["v"], dev["alpha"], dev["beta"], dev_err=err)
    G = torch.from_numpy(dMT).cuda()
    g = sdm.scan_backward(*sel, dev["v"], dev["alpha"], dev["beta"], w_prev, r_rows,
                          torch.from_numpy(dO).cuda(), G)
    dkp = sdm.select_backward(sel[0], g["dsc_w"], S)
    dqp = sdm.select_backward(sel[2], g["dsc_r"], S)
    torch.cuda.synchronize()
    assert err.item() == 0
    return sel, o, M, w_prev, r_rows, g, G, dkp, dqp


def _oracle_backward(host_v, alpha, beta, sel, M0, dO, dMT):
    iw, sw, ir, sr = (x.cpu().numpy() for x in sel)
    B, H, T, W = iw.shape
    R, N, dv = ir.shape[-1], M0.shape[1], M0.shape[2]
    nh = B * H
    Minit = np.broadcast_to(M0[None], (B,) + M0.shape).reshape(nh, N, dv)
    ref = oracle.scan_backward(Minit, iw.reshape(nh, T, W), sw.reshape(nh, T, W), ir.reshape(nh, T, R),
                               sr.reshape(nh, T, R), host_v.reshape(nh, T, dv), alpha.reshape(nh, T),
                               beta.reshape(nh, T), dO.reshape(nh, T, dv), dMT.reshape(nh, N, dv))
    S = int(round(np.sqrt(N)))
    ref["dkp"] = oracle.select_backward(S, iw.reshape(nh, T, W), ref["dsc_w"])
    ref["dqp"] = oracle.select_backward(S, ir.reshape(nh, T, R), ref["dsc_r"])
    return ref


def _check(g, G, dkp, dqp, ref, B, H, label):
    nh = B * H
    for name in ("dv", "dalpha", "dbeta", "dsc_w", "dsc_r"):
        e = normwise(g[name].cpu().numpy().reshape(ref[name].shape), ref[name])
        assert e <= GTOL, f"{label} {name} error {e:.3e}"
    N, dv = ref["dM0"].shape[1:]
    e = normwise(G.cpu().numpy().reshape(nh, N, dv), ref["dM0"])
    assert e <= GTOL, f"{label} dM0 per (b, h) error {e:.3e}"
    shared = ref["dM0"].reshape(B, H, N, dv).sum(axis=0)
    e = normwise(g["dM0"].cpu().numpy(), shared)
    assert e <= GTOL, f"{label} shared dM0 error {e:.3e}"
    for name, x in (("dkp", dkp), ("dqp", dqp)):
        e = normwise(x.cpu().numpy().reshape(ref[name].shape), ref[name])
        assert e <= GTOL, f"{label} {name} error {e:.3e}"


@pytest.mark.parametrize("B,H,T,S,dv,W,R,vdt", [
    (1, 1, 1, 4, 4, 2, 3, torch.float32),          # one token, d_v = 4 (4-column slices)
    (2, 2, 50, 8, 16, 6, 5, torch.float32),        # ragged W, R against the rows per pass
    (1, 3, 97, 6, 24, 9, 20, torch.bfloat16),      # K > S, d_v = 24 (8-column slices)
    (2, 1, 300, 16, 64, 64, 64, torch.bfloat16),   # rows rewritten and reread across tokens
    (1, 2, 40, 4, 32, 16, 16, torch.float32),      # W = R = N: every row every token
])
def test_backward_matches_oracle(B, H, T, S, dv, W, R, vdt):
    rng = np.random.default_rng(B * 1000 + T + dv)
    host, dev, M0, dO, dMT = _random(rng, B, H, T, S, dv, vdt)
    sel, o, M, w_prev, r_rows, g, G, dkp, dqp = _gpu_backward(dev, M0, dO, dMT, W, R)
    ref = _oracle_backward(host["v"], host["alpha"], host["beta"], sel, M0, dO, dMT)
    _check(g, G, dkp, dqp, ref, B, H, (B, H, T, S, dv, W, R))


def test_forward_train_equals_forward_and_keeps_the_rows():
    rng = np.random.default_rng(11)
    B, H, T, S, dv, W, R = 2, 2, 64, 8, 32, 8, 8
    host, dev, M0, dO, dMT = _random(rng, B, H, T, S, dv, torch.float32)
    sel = sdm.select(dev["kp"], dev["qp"], W, R)
    M1 = torch.from_numpy(np.broadcast_to(M0[None], (B,) + M0.shape).copy()).cuda()
    M2 = M1.clone()
    o1 = sdm.scan_forward(M1, *sel, dev["v"], dev["alpha"], dev["beta"])
    o2, w_prev, r_rows = sdm.scan_forward_train(M2, *sel, dev["v"], dev["alpha"], dev["beta"])
    torch.cuda.synchronize()
    assert torch.equal(M1, M2) and torch.equal(o1, o2)
    # token 0's write rows are M_0's rows; the read rows reproduce o
    iw = sel[0].cpu().numpy()
    wp = w_prev.cpu().numpy()
    for b in range(B):
        for h in range(H):
            assert np.array_equal(wp[b, h, 0], M0[h][iw[b, h, 0]])
    r = torch.softmax(sel[3].double(), dim=-1)
    o_rows = torch.einsum("bhtr,bhtrd->bhtd", r, r_rows.double())
    assert float((o_rows - o2.double()).abs().max()) <= 1e-5


OUTPUTS = ("dv", "dalpha", "dbeta", "dsc_w", "dsc_r", "dM0")


@pytest.mark.parametrize("B,H,T,S,dv,W,R,vdt", [
    (1, 1, 1, 4, 4, 2, 3, torch.float32),          # one token: every slot's adjoint is zero
    (2, 2, 50, 8, 16, 6, 5, torch.float32),
    (1, 3, 97, 6, 24, 9, 20, torch.bfloat16),
    (2, 1, 300, 16, 64, 64, 64, torch.bfloat16),   # rows rewritten and reread across tokens
    (1, 2, 40, 4, 32, 16, 16, torch.float32),      # W = R = N: only the last token's read slots are zero
    (3, 1, 70, 12, 8, 40, 33, torch.float32),      # W + R = 73: three words of zero bits, ragged
    (33, 1, 6, 4, 8, 3, 2, torch.float32),         # B > 32: the reduction without per-group masks
])
def test_final_zero_equals_the_cleared_adjoint(B, H, T, S, dv, W, R, vdt):
    """sdm_scan_backward_ex with SDM_BWD_FINAL_ZERO, G filled with NaN on entry, gives the
    values of the full pass with G cleared (torch.equal: equal values, a zero's sign aside),
    twice in a row on one workspace (the previous call's table and bits are stale)."""
    rng = np.random.default_rng(7 * T + W + R)
    host, dev, M0, dO, dMT = _random(rng, B, H, T, S, dv, vdt)
    sel = sdm.select(dev["kp"], dev["qp"], W, R)
    M = torch.from_numpy(np.broadcast_to(M0[None], (B,) + M0.shape).copy()).cuda()
    o, w_prev, r_rows = sdm.scan_forward_train(M, *sel, dev["v"], dev["alpha"], dev["beta"])
    dO_d = torch.from_numpy(dO).cuda()
    N = S * S
    G_ref = torch.zeros((B, H, N, dv), device="cuda")
    ref = sdm.scan_backward(*sel, dev["v"], dev["alpha"], dev["beta"], w_prev, r_rows, dO_d, G_ref)
    ws = torch.empty(sdm.backward_workspace_size(B, H, T, N, dv, W, R, True), dtype=torch.uint8, device="cuda")
    for rep in range(2):
        G = torch.full((B, H, N, dv), float("nan"), device="cuda")
        got = sdm.scan_backward(*sel, dev["v"], dev["alpha"], dev["beta"], w_prev, r_rows, dO_d, G, workspace=ws,
                                final_zero=True)
        torch.cuda.synchronize()
        for name in OUTPUTS:
            assert torch.equal(got[name], ref[name]), (rep, name)
        assert torch.equal(G, G_ref), rep
    # dM0 only: the same outputs; rows of G no slot reads stay as they were (NaN here), and
    # those are exactly the rows whose gradient is zero
    G = torch.full((B, H, N, dv), float("nan"), device="cuda")
    got = sdm.scan_backward(*sel, dev["v"], dev["alpha"], dev["beta"], w_prev, r_rows, dO_d, G, workspace=ws,
                            final_zero=True, dm0_only=True)
    torch.cuda.synchronize()
    for name in OUTPUTS:
        assert torch.equal(got[name], ref[name]), ("dm0_only", name)
    left = torch.isnan(G)
    assert torch.equal(G[~left], G_ref[~left])
    assert bool((G_ref[left] == 0).all())


def test_final_zero_with_no_tokens_clears_the_adjoint():
    B, H, N, dv, W, R = 2, 2, 64, 8, 4, 4
    e = lambda *sh, dt=torch.float32: torch.empty(sh, dtype=dt, device="cuda")
    sel = (e(B, H, 0, W, dt=torch.int32), e(B, H, 0, W), e(B, H, 0, R, dt=torch.int32), e(B, H, 0, R))
    G = torch.full((B, H, N, dv), float("nan"), device="cuda")
    g = sdm.scan_backward(*sel, e(B, H, 0, dv), e(B, H, 0), e(B, H, 0), e(B, H, 0, W, dv), e(B, H, 0, R, dv),
                          e(B, H, 0, dv), G, final_zero=True)
    torch.cuda.synchronize()
    assert torch.equal(G, torch.zeros_like(G))
    assert torch.equal(g["dM0"], torch.zeros_like(g["dM0"]))


@pytest.mark.parametrize("final_zero", [False, True])
def test_backward_on_the_small_workload_sampled_heads(final_zero):
    """B4 H8 T2048 N=65,536 d_v=64 W=R=32, bf16 inputs: the whole backward on the GPU,
    the oracle on two heads (dL/dM_T = 0; with final_zero, G starts as NaN and is ignored)."""
    cfg = wl.B4H8_T2048
    d = device_inputs(cfg)
    M0 = device_M0(cfg)
    sel = sdm.select(d["kp"], d["qp"], cfg.W, cfg.R)
    M = torch.empty((cfg.B, cfg.H, cfg.N, cfg.d_v), device="cuda")
    sdm.init_state_from_M0(M, M0)
    o, w_prev, r_rows = sdm.scan_forward_train(M, *sel, d["v"], d["alpha"], d["beta"])
    rng = np.random.default_rng(21)
    dO = torch.from_numpy(rng.standard_normal((cfg.B, cfg.H, cfg.T, cfg.d_v)).astype(np.float32)).cuda()
    G = torch.full((cfg.B, cfg.H, cfg.N, cfg.d_v), float("nan") if final_zero else 0.0, device="cuda")
    g = sdm.scan_backward(*sel, d["v"], d["alpha"], d["beta"], w_prev, r_rows, dO, G, shared_M0=False,
                          final_zero=final_zero)
    torch.cuda.synchronize()
    M0h = M0.cpu().numpy()
    for b, h in ((0, 0), (cfg.B - 1, cfg.H - 1)):
        s = lambda x: x[b, h].cpu().numpy()[None]
        ref = oracle.scan_backward(M0h[h][None], s(sel[0]), s(sel[1]), s(sel[2]), s(sel[3]),
                                   to_np(d["v"][b, h])[None], s(d["alpha"]), s(d["beta"]), s(dO))
        for name in ("dv", "dalpha", "dbeta", "dsc_w", "dsc_r"):
            e = normwise(g[name][b, h].cpu().numpy()[None], ref[name])
            assert e <= GTOL, (name, b, h, e)
        assert normwise(G[b, h].cpu().numpy()[None], ref["dM0"]) <= GTOL


def test_fill_state_sets_every_entry():
    """sdm_fill_state (the adjoint table cleared before the reverse pass) writes every entry."""
    M = torch.full((2, 3, 1000, 16), float("nan"), device="cuda")
    sdm.fill_state(M, 0.0)
    torch.cuda.synchronize()
    assert torch.equal(M, torch.zeros_like(M))
    sdm.fill_state(M, 1.5)
    torch.cuda.synchronize()
    assert bool((M == 1.5).all())


def test_backward_at_the_benchmark_size():
    """B16 H4 T8192 N=2^20 d_v=128 W=R=128, bf16 inputs, as the backward benchmark runs it
    (zero final adjoint, dM0 only, M_0 shared across the batch): the gradients of two sampled
    sequence-heads against the oracle; dM0 bit for bit equal to the mode that also writes
    each sequence's dL/dM_0, whose sampled sequence-heads match the oracle's dM0."""
    cfg = wl.B16H4_T8192
    d = device_inputs(cfg)
    M0 = device_M0(cfg)
    sel = sdm.select(d["kp"], d["qp"], cfg.W, cfg.R)
    del d["kp"], d["qp"]
    M = torch.empty((cfg.B, cfg.H, cfg.N, cfg.d_v), device="cuda")
    sdm.init_state_from_M0(M, M0)
    o, w_prev, r_rows = sdm.scan_forward_train(M, *sel, d["v"], d["alpha"], d["beta"])
    del o
    rng = np.random.default_rng(23)
    dO = torch.from_numpy(rng.standard_normal((cfg.B, cfg.H, cfg.T, cfg.d_v)).astype(np.float32)).cuda()
    M.fill_(float("nan"))  # the adjoint table: ignored with a zero final adjoint
    G = M
    g = sdm.scan_backward(*sel, d["v"], d["alpha"], d["beta"], w_prev, r_rows, dO, G, shared_M0=True,
                          final_zero=True, dm0_only=True)
    torch.cuda.synchronize()
    heads = ((0, 0), (cfg.B - 1, cfg.H - 1))
    M0h = M0.cpu().numpy()
    refs = {}
    for b, h in heads:
        s = lambda x: x[b, h].cpu().numpy()[None]
        refs[b, h] = oracle.scan_backward(M0h[h][None], s(sel[0]), s(sel[1]), s(sel[2]), s(sel[3]),
                                          to_np(d["v"][b, h])[None], s(d["alpha"]), s(d["beta"]), s(dO))
        for name in ("dv", "dalpha", "dbeta", "dsc_w", "dsc_r"):
            e = normwise(g[name][b, h].cpu().numpy()[None], refs[b, h][name])
            assert e <= GTOL, (name, b, h, e)
    dM0 = g["dM0"].clone()
    G.fill_(float("nan"))
    g2 = sdm.scan_backward(*sel, d["v"], d["alpha"], d["beta"], w_prev, r_rows, dO, G, shared_M0=True,
                           final_zero=True)
    torch.cuda.synchronize()
    assert torch.equal(g2["dM0"], dM0)
    for b, h in heads:
        assert normwise(G[b, h].cpu().numpy()[None], refs[b, h]["dM0"]) <= GTOL
