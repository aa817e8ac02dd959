"""The two selection kernels for bf16 halves: the counting selection (one histogram of exact
values per half and one of the staircase's pair sums, whose prefix sums place every
selected key) and the general one (radix select on composite keys, then a bitonic sort).
Both are forced through sdm_select_tuned and compared with the oracle's top-k, bit for bit
(slots and scores), on inputs that take every branch of the counting kernel: Gaussian
halves (the window holds the top-k), halves with hot indices (the hot-slot workload's
bias), halves whose top-k lie 4-8 binades below a few outliers (the 256-code window holds
too few keys: the fallback), tie-heavy halves (many keys share a value: per-bin ordering,
and more than 32 keys at the cut: the fallback), widely spread halves (the top-k leave the
window: the fallback), constant halves (every key ties) and halves of negative values only.
"""
import numpy as np
import pytest
import torch

import oracle
import sparse_state_linear_sdm_gb300 as sdm
from sparse_state_linear_sdm_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _bf16(x):
    return wl.bf16_to_f32(wl.bf16_bits(np.asarray(x, np.float32)))


def _halves(rng, kind, shape):
    S = shape[-1]
    if kind == "gauss":
        x = rng.standard_normal(shape)
    elif kind == "hot":
        x = rng.standard_normal(shape) + 2.0 * np.exp(-np.arange(S) / 16.0)
    elif kind == "outlier":  # a few entries far above the rest
        x = 0.1 * rng.standard_normal(shape) * np.exp2(rng.integers(-2, 3, size=shape[:-1] + (1,)))
        idx = rng.integers(0, S, size=shape[:-1] + (3,))
        np.put_along_axis(x, idx, 8.0, axis=-1)
    elif kind == "ties":
        vals = np.array([-2.0, -1.0, -0.5, -0.0, 0.0, 0.5, 1.0, 1.5, 2.0])
        x = vals[rng.integers(0, len(vals), size=shape)]
    elif kind == "spread":   # |x| over many binades: few keys per 256-code window
        x = rng.standard_normal(shape) * np.exp2(rng.integers(-40, 40, size=shape))
    elif kind == "const":
        x = np.full(shape, 0.75)
    elif kind == "negative":
        x = -np.abs(rng.standard_normal(shape)) - 0.01
    else:
        raise ValueError(kind)
    return _bf16(x)


SHAPES = [(8, 8, 8), (8, 64, 64), (16, 40, 16), (24, 100, 128), (32, 8, 8), (64, 100, 64),
          (256, 32, 128), (512, 64, 64), (1024, 128, 128), (1024, 1, 128), (1024, 128, 5)]
KINDS = ["gauss", "hot", "outlier", "ties", "spread", "const", "negative"]


@pytest.mark.parametrize("S,W,R", SHAPES)
@pytest.mark.parametrize("kind", KINDS)
def test_counting_and_general_selection_match_the_oracle(S, W, R, kind):
    rng = np.random.default_rng(S * 131 + W * 7 + R + KINDS.index(kind))
    n = 300
    shape = (1, 1, n, 2, S)
    kp, qp = _halves(rng, kind, shape), _halves(rng, kind, shape)
    kp_d = torch.from_numpy(kp).cuda().to(torch.bfloat16)
    qp_d = torch.from_numpy(qp).cuda().to(torch.bfloat16)
    ow, osw = oracle.select(kp[0, 0], W)
    orr, osr = oracle.select(qp[0, 0], R)
    for path in (sdm.SELECT_COUNTING, sdm.SELECT_GENERAL, sdm.SELECT_AUTO):
        iw, sw, ir, sr = sdm.select(kp_d, qp_d, W, R, path=path)
        torch.cuda.synchronize()
        assert np.array_equal(iw[0, 0].cpu().numpy(), ow), (path, "write slots")
        assert np.array_equal(ir[0, 0].cpu().numpy(), orr), (path, "read slots")
        assert np.array_equal(sw[0, 0].cpu().numpy(), osw), (path, "write scores")
        assert np.array_equal(sr[0, 0].cpu().numpy(), osr), (path, "read scores")


def test_counting_selection_limits():
    """Outside its limits the counting kernel is refused, and the automatic choice falls back."""
    x = torch.zeros((1, 1, 4, 2, 12), dtype=torch.bfloat16, device="cuda")   # S % 8 != 0
    with pytest.raises(sdm.SDMError):
        sdm.select(x, x, 4, 4, path=sdm.SELECT_COUNTING)
    sdm.select(x, x, 4, 4, path=sdm.SELECT_AUTO)
    y = torch.zeros((1, 1, 4, 2, 64), dtype=torch.float32, device="cuda")    # fp32 halves
    with pytest.raises(sdm.SDMError):
        sdm.select(y, y, 4, 4, path=sdm.SELECT_COUNTING)
    z = torch.zeros((1, 1, 4, 2, 64), dtype=torch.bfloat16, device="cuda")   # W > 128
    with pytest.raises(sdm.SDMError):
        sdm.select(z, z, 200, 4, path=sdm.SELECT_COUNTING)
    torch.cuda.synchronize()


def test_counting_selection_on_the_default_workload_shape():
    """B16 H4 S=1024 W=R=128, 512 tokens drawn by the device generator: the automatic path
    (the counting kernel) equals the general kernel bit for bit, and the oracle on a head."""
    cfg = wl.B16H4_T8192
    T = 512
    d = sdm.gen_inputs(cfg.seed, cfg.B, cfg.H, T, cfg.S, cfg.d_v, torch.bfloat16, cfg.alpha_lo, 1,
                       T_total=cfg.T, device="cuda")
    a = sdm.select(d["kp"], d["qp"], cfg.W, cfg.R, path=sdm.SELECT_AUTO)
    g = sdm.select(d["kp"], d["qp"], cfg.W, cfg.R, path=sdm.SELECT_GENERAL)
    torch.cuda.synchronize()
    for x, y in zip(a, g):
        assert torch.equal(x, y)
    host = wl.inputs(cfg, 5, 6, 2, 3, 0, T)
    ow, _ = oracle.select(host["kp"][0, 0], cfg.W)
    orr, _ = oracle.select(host["qp"][0, 0], cfg.R)
    assert np.array_equal(a[0][5, 2].cpu().numpy(), ow)
    assert np.array_equal(a[2][5, 2].cpu().numpy(), orr)
