"""Long-context stream: B=1, H=4, N=1,048,576, d_v=128, W=R=128, T=1,048,576 tokens fed
in 65,536-token chunks drawn in HBM by the counter-based generator, the state carried
across chunks (constant state, arbitrarily long sequences: "Significato e
Rivendicazioni" of the Sparse Delta Memory technical summary).

The oracle recomputes one head over the whole first chunk (every output and the final
state of that head) and, at depth, over the whole last chunk: started from the GPU's state
of that head after 983,040 tokens, every output of the last 65,536 tokens and the state
after the 1,048,576th token are compared; properties that hold at any length cover the
rest (chunked = unchunked, bit for bit).
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_state_linear_sdm_gb300 as sdm
from sparse_state_linear_sdm_gb300 import workloads as wl

from sdm_testlib import TOL, device_M0, scaled_err, to_np

pytestmark = pytest.mark.gpu

CFG = wl.STREAM_B1H4_T1M


def _chunk(t_off, T):
    return sdm.gen_inputs(CFG.seed, CFG.B, CFG.H, T, CFG.S, CFG.d_v, torch.bfloat16, CFG.alpha_lo, 1,
                          t_off=t_off, T_total=CFG.T, device="cuda")


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_stream_generator_chunks_match_the_whole_sequence():
    whole = _chunk(0, 2048)
    parts = [_chunk(0, 1000), _chunk(1000, 1048)]
    for k in whole:
        assert torch.equal(whole[k], torch.cat([p[k] for p in parts], dim=2)), k
    # and the host generator agrees with the device at the far end of the sequence
    d = _chunk(CFG.T - 16, 16)
    host = wl.inputs(CFG, 0, 1, 3, 4, CFG.T - 16, CFG.T)
    for k in ("kp", "qp", "v", "alpha", "beta"):
        assert np.array_equal(to_np(d[k][0, 3]), host[k][0, 0]), k


def test_stream_first_and_last_chunk_against_oracle():
    C = CFG.chunk
    n_chunks = CFG.T // C
    M0 = device_M0(CFG)
    M = torch.empty((1, CFG.H, CFG.N, CFG.d_v), device="cuda")
    sdm.init_state_from_M0(M, M0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = sdm.scan_workspace(1, CFG.H, C, CFG.d_v, CFG.W, CFG.R, "cuda")
    first = None
    for c in range(n_chunks):
        d = _chunk(c * C, C)
        sel = sdm.select(d["kp"], d["qp"], CFG.W, CFG.R)
        if c == n_chunks - 1:
            M_deep = M[0, 0].cpu()   # head 0's state after (n_chunks - 1) * C tokens
        o = sdm.scan_forward(M, *sel, d["v"], d["alpha"], d["beta"], workspace=ws, dev_err=err)
        if c == 0:
            first = (o[0, 0].cpu(), M[0, 0].cpu(), sel[0][0, 0].cpu(), sel[2][0, 0].cpu())
        last = (sel, d, o[0, 0].cpu(), M[0, 0].cpu())
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.isfinite(M).all()

    # head 0 over the whole first chunk
    host = wl.inputs(CFG, 0, 1, 0, 1, 0, C)
    ref = oracle.forward(host["kp"][0], host["qp"][0], host["v"][0], host["alpha"][0], host["beta"][0],
                         wl.initial_state(CFG, 0, 1), CFG.W, CFG.R)
    o0, M00, iw0, ir0 = first
    assert np.array_equal(iw0.numpy(), ref["idx_w"][0])
    assert np.array_equal(ir0.numpy(), ref["idx_r"][0])
    assert scaled_err(o0.numpy(), ref["o"][0]) <= TOL
    assert scaled_err(M00.numpy(), ref["M"][0]) <= TOL

    # head 0 over the whole last chunk, from the GPU's state after (n_chunks - 1) * C tokens
    sel, d, o_last, M_last = last
    t0 = (n_chunks - 1) * C
    host = wl.inputs(CFG, 0, 1, 0, 1, t0, CFG.T)
    ref = oracle.forward(host["kp"][0], host["qp"][0], host["v"][0], host["alpha"][0], host["beta"][0],
                         M_deep.numpy()[None], CFG.W, CFG.R)
    assert np.array_equal(sel[0][0, 0].cpu().numpy(), ref["idx_w"][0])
    assert np.array_equal(sel[2][0, 0].cpu().numpy(), ref["idx_r"][0])
    assert np.array_equal(sel[1][0, 0].cpu().numpy(), ref["sc_w"][0])
    assert np.array_equal(sel[3][0, 0].cpu().numpy(), ref["sc_r"][0])
    assert scaled_err(o_last.numpy(), ref["o"][0]) <= TOL
    assert scaled_err(M_last.numpy(), ref["M"][0]) <= TOL

    # selection of the last tokens of another head (pure per token)
    h, n = 2, 64
    kp = wl.halves(CFG, wl.FIELD_KP, 0, 1, h, h + 1, CFG.T - n, CFG.T)[0, 0]
    qp = wl.halves(CFG, wl.FIELD_QP, 0, 1, h, h + 1, CFG.T - n, CFG.T)[0, 0]
    rw, _ = oracle.select(kp, CFG.W)
    rr, _ = oracle.select(qp, CFG.R)
    assert np.array_equal(sel[0][0, h, C - n:].cpu().numpy(), rw)
    assert np.array_equal(sel[2][0, h, C - n:].cpu().numpy(), rr)


def test_stream_chunked_equals_one_call():
    C = 4096
    M0 = device_M0(CFG)
    d = _chunk(0, 2 * C)
    sel = sdm.select(d["kp"], d["qp"], CFG.W, CFG.R)
    M1 = torch.empty((1, CFG.H, CFG.N, CFG.d_v), device="cuda")
    sdm.init_state_from_M0(M1, M0)
    o1 = sdm.scan_forward(M1, *sel, d["v"], d["alpha"], d["beta"])
    M2 = torch.empty_like(M1)
    sdm.init_state_from_M0(M2, M0)
    outs = []
    for c in range(2):
        part = [x[:, :, c * C:(c + 1) * C].contiguous() for x in sel]
        outs.append(sdm.scan_forward(M2, *part, *[d[k][:, :, c * C:(c + 1) * C].contiguous()
                                                   for k in ("v", "alpha", "beta")]))
    assert torch.equal(M1, M2)
    assert torch.equal(o1, torch.cat(outs, dim=2))
