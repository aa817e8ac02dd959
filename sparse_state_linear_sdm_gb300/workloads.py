"""Seeded synthetic workloads for the SDM forward path (host side, numpy).

This module holds no part of the method's arithmetic: it only defines the
benchmark/test configurations and draws their inputs.  Both the CUDA path's
tests and the CPU oracle take their inputs from here; the CUDA library carries a
bit-identical device twin of the same generator (``sdm_gen_inputs``) so that
large configurations can be drawn in HBM directly.

Generator ("counter-based", one draw per tensor element):
  * Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
    as 1, 2, 3", SC'11), key = (seed mod 2^32, seed div 2^32), counter =
    (e mod 2^32, e div 2^32, field, 0) where e is the element's row-major index
    in the full logical tensor and field names the tensor (FIELD_* below).
  * uniform u1 = ((x0 >> 8) + 1) * 2^-24 in (0, 1] from the first output word;
    k = x1 >> 8 (24 bits) from the second sets the Box-Muller angle 2*pi*k/2^24.
  * normal z = sqrt(-2 ln u1) * cos(2*pi*k/2^24) (Box and Muller, 1958), with ln,
    cos, sin and exp evaluated by the fixed series below using only
    correctly-rounded fp32 +, -, *, / and sqrt, so that any IEEE machine gives the
    same bits.  ln u = e ln2 + 2 atanh((f-1)/(f+1)) for u = f 2^e,
    f in [sqrt(1/2), sqrt(2)); cos/sin are Taylor series on [0, pi/2) after an
    exact quadrant split of k; exp is 2^n times a Taylor series on |r| <= ln2/2,
    with r = (x - n ln2_hi) - n ln2_lo: ln2 split in a high part with trailing zero
    bits (so n ln2_hi is exact) and the rest, the argument reduction of Cody and
    Waite ("Software Manual for the Elementary Functions", 1980).
  * bf16 fields are rounded from fp32 to nearest-even.
"""
from __future__ import annotations

import ctypes
import dataclasses
import math
import os
import subprocess
import threading

import numpy as np

FIELD_KP, FIELD_QP, FIELD_V, FIELD_ALPHA, FIELD_BETA, FIELD_M0 = 0, 1, 2, 3, 4, 5
FIELD_X, FIELD_WKQ = 6, 7

_MASK = np.uint64(0xFFFFFFFF)
_PM0 = np.uint64(0xD2511F53)
_PM1 = np.uint64(0xCD9E8D57)
_PW0 = 0x9E3779B9
_PW1 = 0xBB67AE85


def _f(bits):
    return np.uint32(bits).view(np.float32)


# fp32 constants, given by their bit patterns (identical in the CUDA twin)
LN2 = _f(0x3F317218)
SQRT2 = _f(0x3FB504F3)
_LNC = [_f(0x3DE38E39), _f(0x3E124925), _f(0x3E4CCCCD), _f(0x3EAAAAAB)]  # 1/9, 1/7, 1/5, 1/3
ANGLE_STEP = _f(0x34C90FDB)  # (pi/2) / 2^22
_SINC = [_f(0x2F309231), _f(0xB2D7322B), _f(0x3638EF1D), _f(0xB9500D01), _f(0x3C088889),
         _f(0xBE2AAAAB)]  # 1/13!, -1/11!, 1/9!, -1/7!, 1/5!, -1/3!
_COSC = [_f(0xAD49CBA5), _f(0x310F76C7), _f(0xB493F27E), _f(0x37D00D01), _f(0xBAB60B61),
         _f(0x3D2AAAAB), _f(0xBF000000)]  # -1/14!, 1/12!, -1/10!, 1/8!, -1/6!, 1/4!, -1/2!
LOG2E = _f(0x3FB8AA3B)
LN2_HI = _f(0x3F317200)
LN2_LO = _f(0x35BFBE8E)
_EXPC = [_f(0x37D00D01), _f(0x39500D01), _f(0x3AB60B61), _f(0x3C088889), _f(0x3D2AAAAB),
         _f(0x3E2AAAAB), _f(0x3F000000)]  # 1/8!, 1/7!, ..., 1/2!
_ONE = np.float32(1.0)
_HALF = np.float32(0.5)
_TWO = np.float32(2.0)
_MTWO = np.float32(-2.0)
_2M24 = np.float32(2.0 ** -24)


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Philox4x32 with 10 rounds.  c*: uint32-valued arrays; k0, k1: 32-bit key words."""
    c0, c1, c2, c3 = (np.asarray(c, np.uint64) for c in (c0, c1, c2, c3))
    for r in range(10):
        if r:
            k0 = (k0 + _PW0) & 0xFFFFFFFF
            k1 = (k1 + _PW1) & 0xFFFFFFFF
        p0 = c0 * _PM0
        p1 = c2 * _PM1
        c0, c1, c2, c3 = ((p1 >> np.uint64(32)) ^ c1 ^ np.uint64(k0), p1 & _MASK,
                          (p0 >> np.uint64(32)) ^ c3 ^ np.uint64(k1), p0 & _MASK)
    return tuple(c.astype(np.uint32) for c in (c0, c1, c2, c3))


def _words(seed: int, field: int, e):
    e = np.asarray(e, np.uint64)
    x0, x1, _, _ = philox4x32_10(e & _MASK, e >> np.uint64(32), np.full(e.shape, field, np.uint64),
                                 np.zeros(e.shape, np.uint64), seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    return x0, x1


def _uniform_open(x0):
    return ((x0 >> np.uint32(8)).astype(np.float32) + _ONE) * _2M24  # (0, 1]


def _ln(u):
    """Natural log of fp32 u in (0, 1] with fixed fp32 operations."""
    bits = u.view(np.uint32)
    e = (bits >> np.uint32(23)).astype(np.int32) - 127
    f = ((bits & np.uint32(0x7FFFFF)) | np.uint32(0x3F800000)).view(np.float32)
    big = f > SQRT2
    f = np.where(big, f * _HALF, f).astype(np.float32)
    e = e + big.astype(np.int32)
    z = (f - _ONE) / (f + _ONE)
    z2 = z * z
    p = _LNC[0]
    for c in _LNC[1:]:
        p = p * z2 + c
    p = p * z2 + _ONE
    t = z * p
    return e.astype(np.float32) * LN2 + (t + t)


def _cos_turn(k24):
    """cos(2*pi*k/2^24) for 24-bit integers k, with fixed fp32 operations."""
    k24 = k24.astype(np.uint32)
    quad = k24 >> np.uint32(22)
    phi = (k24 & np.uint32(0x3FFFFF)).astype(np.float32) * ANGLE_STEP
    p2 = phi * phi
    s = _SINC[0]
    for c in _SINC[1:]:
        s = s * p2 + c
    s = phi * (s * p2 + _ONE)
    c_ = _COSC[0]
    for c in _COSC[1:]:
        c_ = c_ * p2 + c
    c_ = c_ * p2 + _ONE
    out = np.where(quad == 0, c_, np.where(quad == 1, -s, np.where(quad == 2, -c_, s)))
    return out.astype(np.float32)


def _exp(x):
    """exp(x) for moderate fp32 x (|x| < 80) with fixed fp32 operations."""
    n = np.floor(x * LOG2E + _HALF).astype(np.float32)
    r = (x - n * LN2_HI) - n * LN2_LO
    p = _EXPC[0]
    for c in _EXPC[1:]:
        p = p * r + c
    p = (p * r + _ONE) * r + _ONE
    scale = ((n.astype(np.int32) + 127).astype(np.uint32) << np.uint32(23)).view(np.float32)
    return (p * scale).astype(np.float32)


def normal(seed: int, field: int, e):
    """Standard normal fp32 draws for element indices e (uint64-valued array)."""
    x0, x1 = _words(seed, field, e)
    r = np.sqrt(_MTWO * _ln(_uniform_open(x0))).astype(np.float32)
    return (r * _cos_turn(x1 >> np.uint32(8))).astype(np.float32)


def uniform(seed: int, field: int, e):
    """Uniform fp32 draws in (0, 1] for element indices e."""
    x0, _ = _words(seed, field, e)
    return _uniform_open(x0)


_HERE = os.path.dirname(os.path.abspath(__file__))
_FAST_SRC = os.path.join(_HERE, "workloads_gen.c")
_FAST_SO = os.path.join(_HERE, "_build", "libsdm_workloads.so")
_fast_lock = threading.Lock()
_fast_lib = None


def build_fast(force: bool = False) -> str:
    """Compile the threaded C fast path of this generator (same bits as the numpy one)."""
    if not force and os.path.exists(_FAST_SO) and os.path.getmtime(_FAST_SO) >= os.path.getmtime(_FAST_SRC):
        return _FAST_SO
    os.makedirs(os.path.dirname(_FAST_SO), exist_ok=True)
    tmp = _FAST_SO + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
                    "-fno-fast-math", "-o", tmp, _FAST_SRC, "-lm"], check=True)
    os.replace(tmp, _FAST_SO)
    return _FAST_SO


def _fast():
    global _fast_lib
    with _fast_lock:
        if _fast_lib is None:
            lib = ctypes.CDLL(build_fast())
            lib.sdm_workloads_fill.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_uint64, ctypes.c_int64,
                                               ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
            lib.sdm_workloads_fill.restype = ctypes.c_int
            _fast_lib = lib
    return _fast_lib


def fill_range(seed: int, field: int, e0: int, n: int, kind: str = "normal", n_threads=None):
    """Draws for the contiguous element indices e0 .. e0+n-1 (fp32 [n]); kind "normal"
    or "uniform".  Threaded C; bit-identical to normal()/uniform()."""
    out = np.empty(int(n), np.float32)
    nt = int(n_threads) if n_threads else (os.cpu_count() or 1)
    _fast().sdm_workloads_fill(seed, field, e0, int(n), 0 if kind == "normal" else 1, out.ctypes.data, nt)
    return out


def sigmoid_fixed(z):
    return (_ONE / (_ONE + _exp(-z))).astype(np.float32)


def bf16_bits(x):
    """Round fp32 to bf16 (nearest-even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)).astype(np.uint16)


def bf16_to_f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass(frozen=True)
class SDMConfig:
    """One synthetic SDM forward workload.  S = sqrt(N) is the length of each
    key/query half; W/R are the write/read slot counts per token."""
    name: str
    B: int
    H: int
    T: int
    S: int
    d_v: int
    W: int
    R: int
    in_dtype: str          # "f32" or "bf16" for k', q', v
    alpha_lo: float        # alpha ~ U(alpha_lo, 1)
    beta_kind: str         # "uniform" (U(0,1)) or "sigmoid" (sigmoid of N(0,1))
    hot_bias: bool         # add 2*exp(-j/16) to index j of every half
    seed: int
    chunk: int | None = None   # streamed in chunks of this many tokens

    @property
    def N(self) -> int:
        return self.S * self.S

    @property
    def head_tokens(self) -> int:
        return self.B * self.H * self.T


TINY_F32 = SDMConfig("tiny-B1H1-T64-N1024-dv16-W8", 1, 1, 64, 32, 16, 8, 8, "f32", 0.9, "uniform",
                     False, 0)
B4H8_T2048 = SDMConfig("B4H8-T2048-N65536-dv64-W32", 4, 8, 2048, 256, 64, 32, 32, "bf16", 0.95,
                       "sigmoid", False, 1)
B8H16_T4096_HOT = SDMConfig("B8H16-T4096-N262144-dv64-W64-hot", 8, 16, 4096, 512, 64, 64, 64, "bf16",
                            0.95, "sigmoid", True, 2)
B16H4_T8192 = SDMConfig("B16H4-T8192-N1M-dv128-W128", 16, 4, 8192, 1024, 128, 128, 128, "bf16", 0.97,
                        "sigmoid", False, 3)
STREAM_B1H4_T1M = SDMConfig("stream-B1H4-T1M-N1M-dv128-W128", 1, 4, 1 << 20, 1024, 128, 128, 128, "bf16",
                            0.97, "sigmoid", False, 4, chunk=65536)

# The workloads in a fixed order (bench.py --config I picks one by position; the seed of
# each is its position).
CONFIGS = [TINY_F32, B4H8_T2048, B8H16_T4096_HOT, B16H4_T8192, STREAM_B1H4_T1M]


def by_name(name: str) -> SDMConfig:
    """The workload with this name."""
    for c in CONFIGS:
        if c.name == name:
            return c
    raise KeyError(name)


def half_bias(cfg: SDMConfig):
    """Per-index bias added to every half (hot slots), fp32 [S], or None."""
    if not cfg.hot_bias:
        return None
    return np.array([2.0 * math.exp(-j / 16.0) for j in range(cfg.S)], np.float64).astype(np.float32)


def _rows(cfg, field, b0, b1, h0, h1, t0, t1, width, kind="normal"):
    """Draws for the [nb, nh, nt, width] box whose elements are e = bht * width + k,
    bht = (b*H + h)*T + t: one contiguous range per (b, h)."""
    out = np.empty((b1 - b0, h1 - h0, t1 - t0, width), np.float32)
    for bi, b in enumerate(range(b0, b1)):
        for hi, h in enumerate(range(h0, h1)):
            e0 = ((b * cfg.H + h) * cfg.T + t0) * width
            out[bi, hi] = fill_range(cfg.seed, field, e0, (t1 - t0) * width, kind).reshape(t1 - t0, width)
    return out


def _bht_index(cfg, b0, b1, h0, h1, t0, t1):
    b = np.arange(b0, b1, dtype=np.uint64)[:, None, None]
    h = np.arange(h0, h1, dtype=np.uint64)[None, :, None]
    t = np.arange(t0, t1, dtype=np.uint64)[None, None, :]
    return (b * np.uint64(cfg.H) + h) * np.uint64(cfg.T) + t      # [nb, nh, nt]


def halves(cfg: SDMConfig, field: int, b0, b1, h0, h1, t0, t1):
    """k' (FIELD_KP) or q' (FIELD_QP) halves for the box b0:b1, h0:h1, t0:t1.

    Returns fp32 [nb, nh, nt, 2, S] holding the exact values the path sees (already
    rounded to bf16 for bf16 configurations)."""
    x = _rows(cfg, field, b0, b1, h0, h1, t0, t1, 2 * cfg.S).reshape(b1 - b0, h1 - h0, t1 - t0, 2, cfg.S)
    bias = half_bias(cfg)
    if bias is not None:
        x = (x + bias).astype(np.float32)
    if cfg.in_dtype == "bf16":
        x = bf16_to_f32(bf16_bits(x))
    return x


def values(cfg: SDMConfig, b0, b1, h0, h1, t0, t1):
    """v [nb, nh, nt, d_v] (fp32 holding bf16-rounded values for bf16 configs)."""
    x = _rows(cfg, FIELD_V, b0, b1, h0, h1, t0, t1, cfg.d_v)
    if cfg.in_dtype == "bf16":
        x = bf16_to_f32(bf16_bits(x))
    return x


def gates(cfg: SDMConfig, b0, b1, h0, h1, t0, t1):
    """(alpha, beta), each fp32 [nb, nh, nt]."""
    lo = np.float32(cfg.alpha_lo)
    u = _rows(cfg, FIELD_ALPHA, b0, b1, h0, h1, t0, t1, 1, "uniform")[..., 0]
    alpha = (lo + (_ONE - lo) * u).astype(np.float32)
    if cfg.beta_kind == "uniform":
        beta = _rows(cfg, FIELD_BETA, b0, b1, h0, h1, t0, t1, 1, "uniform")[..., 0]
    else:
        beta = sigmoid_fixed(_rows(cfg, FIELD_BETA, b0, b1, h0, h1, t0, t1, 1)[..., 0])
    return alpha, beta


M0_SCALE = np.float32(0.02)


def initial_state(cfg: SDMConfig, h0, h1, n0=0, n1=None):
    """Learned-initial-state stand-in M_0 ~ N(0, 0.02^2): fp32 [nh, n1-n0, d_v]."""
    n1 = cfg.N if n1 is None else n1
    out = np.empty((h1 - h0, n1 - n0, cfg.d_v), np.float32)
    for hi, h in enumerate(range(h0, h1)):
        z = fill_range(cfg.seed, FIELD_M0, (h * cfg.N + n0) * cfg.d_v, (n1 - n0) * cfg.d_v)
        out[hi] = (M0_SCALE * z).reshape(n1 - n0, cfg.d_v)
    return out


def inputs(cfg: SDMConfig, b0=0, b1=None, h0=0, h1=None, t0=0, t1=None):
    """All per-token inputs for a box: dict(kp, qp, v, alpha, beta) as fp32 arrays
    with a leading [nb, nh, nt] shape."""
    b1 = cfg.B if b1 is None else b1
    h1 = cfg.H if h1 is None else h1
    t1 = cfg.T if t1 is None else t1
    alpha, beta = gates(cfg, b0, b1, h0, h1, t0, t1)
    return dict(kp=halves(cfg, FIELD_KP, b0, b1, h0, h1, t0, t1),
                qp=halves(cfg, FIELD_QP, b0, b1, h0, h1, t0, t1),
                v=values(cfg, b0, b1, h0, h1, t0, t1), alpha=alpha, beta=beta)


# Projection workload: token features x [B, T, D] and key/query weights w [4*H*S, D].  The
# pages give no model width; D = 2,048 is taken as a width typical of the smallest model
# scale they train (1.4B parameters).  x ~ N(0, 1); w ~ N(0, 1/D) (the usual fan-in
# scaling), so that each projected sub-score is ~ N(0, 1) like the selection workloads'.
PROJ_D = 2048


def projection_features(seed: int, B: int, T: int, D: int, m0: int = 0, m1=None):
    """bf16 bit patterns of x rows m0 .. m1-1 (m = b*T + t) of x [B, T, D]: uint16 [m1-m0, D]."""
    m1 = B * T if m1 is None else m1
    z = fill_range(seed, FIELD_X, m0 * D, (m1 - m0) * D)
    return bf16_bits(z).reshape(m1 - m0, D)


def projection_weights(seed: int, H: int, S: int, D: int):
    """bf16 bit patterns of w [4*H*S, D] ~ N(0, 1/D)."""
    z = fill_range(seed, FIELD_WKQ, 0, 4 * H * S * D)
    scale = np.float32(1.0 / math.sqrt(D))
    return bf16_bits((z * scale).astype(np.float32)).reshape(4 * H * S, D)
