"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI,
run the CPU oracle on the same seeded inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import sparse_state_linear_sdm_gb300 as sdm
from sparse_state_linear_sdm_gb300 import workloads as wl

TOL = 2e-4  # max |x_gpu - x_ref| <= TOL * (1 + |x_ref|), fp32 state vs fp64 oracle


def scaled_err(got, want) -> float:
    g = np.asarray(got, np.float64)
    w = np.asarray(want, np.float64)
    assert g.shape == w.shape, (g.shape, w.shape)
    if g.size == 0:
        return 0.0
    return float((np.abs(g - w) / (1.0 + np.abs(w))).max())


def torch_dtype(cfg):
    return torch.bfloat16 if cfg.in_dtype == "bf16" else torch.float32


def device_inputs(cfg, T=None, t_off=0, device="cuda"):
    """The configuration's inputs drawn in HBM by the device generator."""
    T = cfg.T if T is None else T
    bias = wl.half_bias(cfg)
    bias_d = None if bias is None else torch.from_numpy(bias).to(device)
    return sdm.gen_inputs(cfg.seed, cfg.B, cfg.H, T, cfg.S, cfg.d_v, torch_dtype(cfg), cfg.alpha_lo,
                          0 if cfg.beta_kind == "uniform" else 1, half_bias=bias_d, t_off=t_off,
                          T_total=cfg.T, device=device)


def device_M0(cfg, device="cuda"):
    return sdm.gen_M0(cfg.seed, cfg.H, cfg.N, cfg.d_v, float(wl.M0_SCALE), device=device)


def host_heads(cfg, heads, t0=0, t1=None):
    """Host-generated inputs of the listed (b, h) pairs, stacked: kp/qp [nh, T, 2, S],
    v [nh, T, d_v], alpha/beta [nh, T], M0 [nh, N, d_v] (fp32)."""
    t1 = cfg.T if t1 is None else t1
    parts = [wl.inputs(cfg, b, b + 1, h, h + 1, t0, t1) for b, h in heads]
    out = {k: np.concatenate([p[k].reshape((1,) + p[k].shape[2:]) for p in parts]) for k in parts[0]}
    out["M0"] = np.concatenate([wl.initial_state(cfg, h, h + 1) for _, h in heads])
    return out


def oracle_heads(cfg, host, W=None, R=None):
    W = cfg.W if W is None else W
    R = cfg.R if R is None else R
    return oracle.forward(host["kp"], host["qp"], host["v"], host["alpha"], host["beta"], host["M0"], W, R)


def to_np(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return wl.bf16_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.cpu().numpy()


def check_against_oracle(cfg, heads, o, M, sel, ref, label=""):
    """Compare GPU results of the listed heads (taken from full [B,H,...] tensors)
    with the oracle's: slots bit-exact, scores equal, o and M within TOL."""
    iw, sw, ir, sr = sel
    for k, (b, h) in enumerate(heads):
        g_iw, g_ir = iw[b, h].cpu().numpy(), ir[b, h].cpu().numpy()
        assert np.array_equal(g_iw, ref["idx_w"][k]), f"{label} write slots differ at head {(b, h)}"
        assert np.array_equal(g_ir, ref["idx_r"][k]), f"{label} read slots differ at head {(b, h)}"
        assert np.array_equal(sw[b, h].cpu().numpy(), ref["sc_w"][k]), f"{label} write scores differ"
        assert np.array_equal(sr[b, h].cpu().numpy(), ref["sc_r"][k]), f"{label} read scores differ"
        e_o = scaled_err(o[b, h].cpu().numpy(), ref["o"][k])
        e_m = scaled_err(M[b, h].cpu().numpy(), ref["M"][k])
        assert e_o <= TOL, f"{label} o error {e_o:.3e} at head {(b, h)}"
        assert e_m <= TOL, f"{label} M error {e_m:.3e} at head {(b, h)}"
