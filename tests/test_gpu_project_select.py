"""The projections fused with the selection (sdm_project_select): k' and q' are produced
and reduced to each half's top-k on chip, then the outer top-K runs on the lists.  The
slots and scores must equal, bit for bit, the unfused path on the same inputs:
sdm_project_kq (whose bf16 outputs are checked against the oracle's fp64 projection in
test_gpu_project.py) followed by sdm_select, and the oracle's selection run on those same
bf16 halves.  Shapes cover ragged token blocks (B*T not a multiple of 64), a ragged K block
(D not a multiple of 64), W != R, a single M-tile (S = 128) and the full width (S = 1024,
D = 2048)."""
import numpy as np
import pytest
import torch

import oracle
import sparse_state_linear_sdm_gb300 as sdm
from sparse_state_linear_sdm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


@pytest.mark.parametrize("B,T,D,H,S,W,R", [
    (1, 70, 128, 1, 128, 8, 8),         # one M-tile, one ragged token block
    (2, 300, 256, 2, 256, 32, 20),      # 10 token blocks, the last ragged; W != R
    (1, 64, 72, 1, 512, 64, 128),       # ragged K block (D % 64 != 0)
    (1, 129, 2048, 4, 1024, 128, 128),  # the full-size width and depth
])
def test_fused_projection_selection_equals_project_then_select(B, T, D, H, S, W, R):
    xb = wl.projection_features(B * 17 + T + D, B, T, D).reshape(B, T, D)
    wb = wl.projection_weights(B * 17 + T + D, H, S, D)
    x, w = _bf16_dev(xb), _bf16_dev(wb)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fused = sdm.project_select(x, w, H, S, W, R, dev_err=err)
    kp, qp = sdm.project_kq(x, w, H, S)
    ref = sdm.select(kp, qp, W, R)
    torch.cuda.synchronize()
    assert err.item() == 0
    for name, a, b in zip(("idx_w", "sc_w", "idx_r", "sc_r"), fused, ref):
        assert torch.equal(a, b), name
    # and the oracle's selection on the same bf16 halves, for a few (b, h)
    hk = kp.float().cpu().numpy().reshape(B * H, T, 2, S)
    hq = qp.float().cpu().numpy().reshape(B * H, T, 2, S)
    oiw, osw = oracle.select(hk[:2], W)
    oir, osr = oracle.select(hq[:2], R)
    assert np.array_equal(fused[0].cpu().numpy().reshape(B * H, T, W)[:2], oiw)
    assert np.array_equal(fused[2].cpu().numpy().reshape(B * H, T, R)[:2], oir)
    assert np.array_equal(fused[1].cpu().numpy().reshape(B * H, T, W)[:2], osw)
    assert np.array_equal(fused[3].cpu().numpy().reshape(B * H, T, R)[:2], osr)


def test_fused_projection_selection_limits():
    x = torch.zeros((1, 8, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((4 * 1 * 96, 64), dtype=torch.bfloat16, device="cuda")   # S = 96: S % 128 != 0
    with pytest.raises(sdm.SDMError):
        sdm.project_select(x, w, 1, 96, 8, 8)
    torch.cuda.synchronize()
