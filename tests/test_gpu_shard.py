"""The d_v split on one GPU: the scan of each rank's column slice (shard.scan_dv_slice,
with the full-width selection) gives exactly the matching columns of the full-width scan,
outputs and state, for 2 and 4 slices; the ranks' slices are run one after the other here
(no collective), which is what each rank of a multi-GPU run computes before the
all-gather."""
import numpy as np
import pytest
import torch

import sparse_state_linear_sdm_gb300 as sdm
from sparse_state_linear_sdm_gb300 import shard
from sparse_state_linear_sdm_gb300 import workloads as wl

from sdm_testlib import device_inputs, device_M0

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("world", [2, 4])
@pytest.mark.parametrize("cfg", [wl.B4H8_T2048, wl.B16H4_T8192], ids=lambda c: c.name)
def test_column_slices_reassemble_the_full_scan(cfg, world):
    T = 512
    d = device_inputs(cfg, T=T)
    M0 = device_M0(cfg)
    B = min(cfg.B, 4)
    d = {k: x[:B].contiguous() for k, x in d.items()}
    sel = sdm.select(d["kp"], d["qp"], cfg.W, cfg.R)
    M = torch.empty((B, cfg.H, cfg.N, cfg.d_v), device="cuda")
    sdm.init_state_from_M0(M, M0)
    o = sdm.scan_forward(M, *sel, d["v"], d["alpha"], d["beta"])
    outs = []
    for r in range(world):
        o_loc, M_loc = shard.scan_dv_slice(M0, sel, d["v"], d["alpha"], d["beta"], r, world)
        c0, c1 = shard.dv_columns(cfg.d_v, world, r)
        assert torch.equal(M_loc, M[..., c0:c1]), f"slice {r}: state differs"
        outs.append(o_loc)
        del M_loc
    assert torch.equal(torch.cat(outs, dim=-1), o)
    torch.cuda.synchronize()
