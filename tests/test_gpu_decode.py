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


@pytest.mark.parametrize("graph", [False, True])
def test_decode_steps_equal_one_scan(graph):
    cfg = wl.CONFIGS[1]
    T = 48
    d = device_inputs(cfg, T=T)
    M0 = device_M0(cfg)
    o_ref, M_ref, sel = sdm.forward(d["kp"], d["qp"], d["v"], d["alpha"], d["beta"], M0, cfg.W, cfg.R)
    M = torch.empty_like(M_ref)
    sdm.init_state_from_M0(M, M0)
    step = sdm.DecodeStep(M, cfg.W, cfg.R, in_dtype=torch.bfloat16)
    if graph:
        step.capture()
    outs = []
    for t in range(T):
        o = step(d["kp"][:, :, t:t + 1], d["qp"][:, :, t:t + 1], d["v"][:, :, t:t + 1],
                 d["alpha"][:, :, t:t + 1], d["beta"][:, :, t:t + 1])
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
