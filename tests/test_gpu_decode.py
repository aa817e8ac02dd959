"""Single-token decode with resident state (the inference path): one token per step for
a batch of sequences, replayed from a CUDA graph.  Chaining T decode steps must give
bit for bit what one scan over the T tokens gives, and that matches the oracle."""
import numpy as np
import pytest
import torch

import sparse_state_linear_sdm_gb300 as sdm
from sparse_state_linear_sdm_gb300 import workloads as wl

from sdm_testlib import TOL, device_inputs, device_M0, host_heads, oracle_heads, scaled_err

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("graph,contiguous", [(False, False), (True, False), (True, True)],
                         ids=["copies", "copies+graph", "direct"])
def test_decode_steps_equal_one_scan(graph, contiguous):
    """Token slices of [B, H, T, ...] inputs are strided: they are copied into the step's
    buffers (then the captured graph or a plain launch runs).  Contiguous per-token inputs
    are read where they are by one launch of the single kernel."""
    cfg = wl.B4H8_T2048
    T = 48
    d = device_inputs(cfg, T=T)
    M0 = device_M0(cfg)
    o_ref, M_ref, sel = sdm.forward(d["kp"], d["qp"], d["v"], d["alpha"], d["beta"], M0, cfg.W, cfg.R)
    M = torch.empty_like(M_ref)
    sdm.init_state_from_M0(M, M0)
    step = sdm.DecodeStep(M, cfg.W, cfg.R, in_dtype=torch.bfloat16)
    assert step.fused
    if graph:
        step.capture()
    outs = []
    for t in range(T):
        args = [d[k][:, :, t:t + 1] for k in ("kp", "qp", "v", "alpha", "beta")]
        if contiguous:
            args = [a.contiguous() for a in args]
        assert all(a.is_contiguous() for a in args) == contiguous
        o = step(*args)
        outs.append(o.clone())
    torch.cuda.synchronize()
    assert step.err.item() == 0
    assert torch.equal(M, M_ref)
    assert torch.equal(torch.cat(outs, dim=2), o_ref)
    # and against the oracle on two heads
    heads = [(0, 0), (3, 7)]
    ref = oracle_heads(cfg, host_heads(cfg, heads, 0, T))
    for k, (b, h) in enumerate(heads):
        assert scaled_err(torch.cat(outs, dim=2)[b, h].cpu().numpy(), ref["o"][k]) <= TOL


def _token(rng, B, H, S, dv, dt):
    f = lambda *sh: torch.from_numpy(rng.standard_normal(sh).astype(np.float32)).cuda()
    return dict(kp=f(B, H, 1, 2, S).to(dt), qp=f(B, H, 1, 2, S).to(dt), v=f(B, H, 1, dv).to(dt),
                alpha=torch.from_numpy(rng.uniform(0.8, 1.0, (B, H, 1)).astype(np.float32)).cuda(),
                beta=torch.from_numpy(rng.uniform(0.0, 1.0, (B, H, 1)).astype(np.float32)).cuda())


@pytest.mark.parametrize("B,H,S,dv,W,R,dt,steps", [
    (2, 3, 32, 32, 16, 16, torch.bfloat16, 5),    # one 32-column slice
    (1, 2, 64, 128, 128, 128, torch.bfloat16, 3),  # the default widths
    (2, 1, 8, 64, 40, 64, torch.float32, 6),      # K > S; W = R = N: every row read is also written
    (1, 1, 24, 96, 200, 150, torch.bfloat16, 2),  # K > 128 (wide sort variant); 3 slices
    (3, 2, 16, 32, 8, 3, torch.float32, 4),
    (16, 8, 32, 32, 16, 16, torch.bfloat16, 2),   # more sequence-heads than SM pairs: no clusters
])
def test_fused_decode_equals_select_then_scan(B, H, S, dv, W, R, dt, steps):
    """sdm_decode_step (one kernel) against sdm_select + sdm_scan_forward on the same token,
    chained over several tokens: slots, scores, o and M bit for bit; the step given the
    prebuilt staircase table (decode_table) too."""
    rng = np.random.default_rng(B * 100 + S + dv + W)
    M0 = torch.from_numpy((0.3 * rng.standard_normal((B, H, S * S, dv))).astype(np.float32)).cuda()
    M1, M2, M3 = M0.clone(), M0.clone(), M0.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    table = sdm.decode_table(W, R, S)
    for _ in range(steps):
        x = _token(rng, B, H, S, dv, dt)
        o1, sel1 = sdm.decode_step(x["kp"], x["qp"], x["v"], x["alpha"], x["beta"], M1, W, R, dev_err=err)
        sel2 = sdm.select(x["kp"], x["qp"], W, R)
        o2 = sdm.scan_forward(M2, *sel2, x["v"], x["alpha"], x["beta"])
        o3, sel3 = sdm.decode_step(x["kp"], x["qp"], x["v"], x["alpha"], x["beta"], M3, W, R, dev_err=err,
                                   table=table)
        torch.cuda.synchronize()
        for a, b, c in zip(sel1, sel2, sel3):
            assert torch.equal(a, b)
            assert torch.equal(c, b)
        assert torch.equal(o1, o2)
        assert torch.equal(o3, o2)
        assert torch.equal(M1, M2)
        assert torch.equal(M3, M2)
    assert err.item() == 0


def test_decode_step_graph_uses_one_kernel_and_matches_the_unfused_step():
    cfg = wl.B4H8_T2048
    T = 6
    d = device_inputs(cfg, T=T)
    M0 = device_M0(cfg)
    Ma = torch.empty((cfg.B, cfg.H, cfg.N, cfg.d_v), device="cuda")
    sdm.init_state_from_M0(Ma, M0)
    Mb = Ma.clone()
    fused = sdm.DecodeStep(Ma, cfg.W, cfg.R, in_dtype=torch.bfloat16).capture()
    plain = sdm.DecodeStep(Mb, cfg.W, cfg.R, in_dtype=torch.bfloat16, fused=False).capture()
    assert fused.fused and not plain.fused
    for t in range(T):
        args = [d[k][:, :, t:t + 1] for k in ("kp", "qp", "v", "alpha", "beta")]
        oa = fused(*args).clone()
        ob = plain(*args).clone()
        assert torch.equal(oa, ob)
    torch.cuda.synchronize()
    assert torch.equal(Ma, Mb)


def test_decode_step_column_slices_follow_the_scan_shape():
    """d_v = 24: the scan kernel takes 4-column slices here, and so does the decode kernel."""
    rng = np.random.default_rng(3)
    M1 = torch.from_numpy(rng.standard_normal((1, 1, 64, 24)).astype(np.float32)).cuda()
    M2 = M1.clone()
    for _ in range(3):
        x = _token(rng, 1, 1, 8, 24, torch.float32)
        o1, s1 = sdm.decode_step(x["kp"], x["qp"], x["v"], x["alpha"], x["beta"], M1, 4, 4)
        s2 = sdm.select(x["kp"], x["qp"], 4, 4)
        o2 = sdm.scan_forward(M2, *s2, x["v"], x["alpha"], x["beta"])
        torch.cuda.synchronize()
        assert all(torch.equal(a, b) for a, b in zip(s1, s2))
        assert torch.equal(o1, o2) and torch.equal(M1, M2)
    assert sdm.DecodeStep(M1, 4, 4, in_dtype=torch.float32).fused


def test_decode_at_the_benchmark_size():
    """The decode step at the size its benchmark runs (B=16, H=4, N=2^20, d_v=128,
    W=R=128, bf16 inputs: clusters of two blocks, the staircase table): three tokens through
    DecodeStep against select + scan_forward on a copy of the state, bit for bit, and o of
    two sequence-heads against the oracle."""
    cfg = wl.B16H4_T8192
    T = 3
    d = device_inputs(cfg, T=T)
    M0 = device_M0(cfg)
    M1 = torch.empty((cfg.B, cfg.H, cfg.N, cfg.d_v), dtype=torch.float32, device="cuda")
    sdm.init_state_from_M0(M1, M0)
    M2 = M1.clone()
    step = sdm.DecodeStep(M1, cfg.W, cfg.R, in_dtype=torch.bfloat16)
    assert step.fused and step.table is not None
    outs = []
    for t in range(T):
        args = [d[k][:, :, t:t + 1].contiguous() for k in ("kp", "qp", "v", "alpha", "beta")]
        outs.append(step(*args).clone())
        sel = sdm.select(args[0], args[1], cfg.W, cfg.R)
        o2 = sdm.scan_forward(M2, *sel, *args[2:])
        torch.cuda.synchronize()
        for a, b in zip(step.sel, sel):
            assert torch.equal(a, b)
        assert torch.equal(outs[-1], o2)
    assert step.err.item() == 0
    assert torch.equal(M1, M2)
    del M2
    heads = [(0, 0), (15, 3)]
    ref = oracle_heads(cfg, host_heads(cfg, heads, 0, T))
    o = torch.cat(outs, dim=2)
    for k, (b, h) in enumerate(heads):
        assert scaled_err(o[b, h].cpu().numpy(), ref["o"][k]) <= TOL
