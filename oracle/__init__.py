"""SDM forward oracle: plain CPU reference of the Sparse Delta Memory forward pass.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product library (``sparse_state_linear_sdm_gb300``) shares no code with it.

What it computes follows the "Sparse Delta Memory (SDM)" technical summary
(gist.science/it/paper/2607.07386), section "Meccanismo Core", items 1-4:
product-key top-W / top-R slot selection through
topk(s1 (+) s2) = topk(topk(s1) (+) topk(s2)), the gated delta write
M_t[i] = a_t M_{t-1}[i] + b_t k_t^(i) (v_t - a_t M_{t-1}[i]) on the selected rows
only, and a weighted read of the R selected rows after the write.  The
arithmetic lives in ``sdm_oracle.cpp`` (fp32 selection sums, fp64 state).  Also the
linear projections x -> k', q' (``project``, one fp64 library matmul) and the reverse
mode of the scan and of the selection sums (``scan_backward``, ``select_backward``).

Every function here is pinned against things other than itself:
``tests/test_oracle_pins.py`` (brute force over all N slot scores, a hand-worked
two-token example, invariants of the update equations and closed forms),
``tests/test_oracle_backward_pins.py`` (finite differences, an exact linearity
identity) and ``tests/test_oracle_project_pins.py`` (one-hot features, explicit loops
on tiny sizes, linearity).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdm_oracle.cpp")
_SO = os.path.join(_HERE, "_build", "liboracle_sdm.so")
_lock = threading.Lock()
_lib = None


def compile_library(src: str, so: str) -> str:
    """Compile a C++ source of the oracle into a shared library at ``so`` (host code only)."""
    os.makedirs(os.path.dirname(so), exist_ok=True)
    tmp = so + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-o", tmp, src]
    subprocess.run(cmd, check=True)
    os.replace(tmp, so)
    return so


def build(force: bool = False) -> str:
    """Compile the oracle's C++ into a shared library (host code only)."""
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    return compile_library(_SRC, _SO)


def open_library(path: str) -> ctypes.CDLL:
    """Load a compiled oracle library and declare its entry points."""
    lib = ctypes.CDLL(path)
    i64, i32, p = ctypes.c_longlong, ctypes.c_int, ctypes.c_void_p
    lib.oracle_select.argtypes = [p, i64, i32, i32, p, p, i32]
    lib.oracle_select.restype = i32
    lib.oracle_scan.argtypes = [p, i32, i64, i32, i32, i32, i32, p, p, p, p, p, p, p, p, i32]
    lib.oracle_scan.restype = i32
    lib.oracle_scan_backward.argtypes = [p, i32, i64, i32, i32, i32, i32, p, p, p, p, p, p, p,
                                         p, p, p, p, p, p, p, i32]
    lib.oracle_scan_backward.restype = i32
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = open_library(build())
    return _lib


def _threads(n_threads):
    return int(n_threads) if n_threads else (os.cpu_count() or 1)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def select(halves, K: int, n_threads=None):
    """Top-K slots of every item.  halves: float32 [..., 2, S] (half 0, half 1).

    Returns (idx int32 [..., K], sc float32 [..., K]) ordered by (sum desc, flat asc),
    flat = i*S + j with i from half 0.
    """
    h = _c(halves, np.float32)
    S = h.shape[-1]
    lead = h.shape[:-2]
    n = int(np.prod(lead)) if lead else 1
    idx = np.empty(lead + (K,), np.int32)
    sc = np.empty(lead + (K,), np.float32)
    rc = _load().oracle_select(h.ctypes.data, n, S, K, idx.ctypes.data, sc.ctypes.data,
                               _threads(n_threads))
    if rc != 0:
        raise ValueError(f"oracle_select: bad sizes S={S} K={K}")
    return idx, sc


def select_bruteforce(halves, K: int):
    """Same contract as ``select`` but by ranking all S*S slot scores directly.

    Independent of the C++ selection: the N scores fp32(half0[i] + half1[j]) at
    flat = i*S + j are ordered with numpy's lexsort (score desc, flat asc).
    Used only on tiny inputs to pin the product-key identity.
    """
    h = _c(halves, np.float32)
    S = h.shape[-1]
    lead = h.shape[:-2]
    flat_h = h.reshape(-1, 2, S)
    n = flat_h.shape[0]
    if K < 1 or K > S * S:
        raise ValueError(f"select_bruteforce: bad sizes S={S} K={K}")
    idx = np.empty((n, K), np.int32)
    sc = np.empty((n, K), np.float32)
    flat = np.arange(S * S)
    for it in range(n):
        scores = (flat_h[it, 0][:, None] + flat_h[it, 1][None, :]).astype(np.float32).ravel()
        order = np.lexsort((flat, -scores))[:K]
        idx[it] = flat[order]
        sc[it] = scores[order]
    return idx.reshape(lead + (K,)), sc.reshape(lead + (K,))


def scan(M, idx_w, sc_w, idx_r, sc_r, v, alpha, beta, n_threads=None):
    """Recurrent sparse gated-delta scan of nh independent (sequence, head) pairs.

    M: float64 [nh, N, d_v], updated in place (state before -> after the T tokens).
    idx_w/sc_w: [nh, T, W]; idx_r/sc_r: [nh, T, R]; v: [nh, T, d_v];
    alpha/beta: [nh, T].  Returns o float64 [nh, T, d_v].
    """
    if not (isinstance(M, np.ndarray) and M.dtype == np.float64 and M.flags.c_contiguous):
        raise TypeError("M must be a C-contiguous float64 array (updated in place)")
    nh, N, dv = M.shape
    iw, sw = _c(idx_w, np.int32), _c(sc_w, np.float32)
    ir, sr = _c(idx_r, np.int32), _c(sc_r, np.float32)
    vv = _c(v, np.float32)
    a, b = _c(alpha, np.float32), _c(beta, np.float32)
    T, W = iw.shape[1], iw.shape[2]
    R = ir.shape[2]
    o = np.empty((nh, T, dv), np.float64)
    rc = _load().oracle_scan(M.ctypes.data, nh, N, dv, T, W, R, iw.ctypes.data, sw.ctypes.data,
                             ir.ctypes.data, sr.ctypes.data, vv.ctypes.data, a.ctypes.data,
                             b.ctypes.data, o.ctypes.data, _threads(n_threads))
    if rc != 0:
        raise ValueError("oracle_scan: bad sizes or slot index out of range")
    return o


def forward(kp, qp, v, alpha, beta, M_init, W: int, R: int, n_threads=None):
    """Selection then scan for nh (sequence, head) pairs.

    kp, qp: float32 [nh, T, 2, S]; v: [nh, T, d_v]; alpha, beta: [nh, T];
    M_init: [nh, N, d_v] (copied to fp64; the caller's array is not modified).
    Returns dict(idx_w, sc_w, idx_r, sc_r, o (float64), M (float64 final state)).
    """
    idx_w, sc_w = select(kp, W, n_threads)
    idx_r, sc_r = select(qp, R, n_threads)
    M = np.array(M_init, dtype=np.float64, order="C", copy=True)
    o = scan(M, idx_w, sc_w, idx_r, sc_r, v, alpha, beta, n_threads)
    return dict(idx_w=idx_w, sc_w=sc_w, idx_r=idx_r, sc_r=sc_r, o=o, M=M)


def scan_backward(M_init, idx_w, sc_w, idx_r, sc_r, v, alpha, beta, dO, dMT=None, n_threads=None):
    """Reverse-mode derivative of ``scan`` for L = sum_t <dO_t, o_t> + <dMT, M_T>, slots fixed.

    M_init: [nh, N, d_v] state before token 0 (not modified); dO: [nh, T, d_v];
    dMT: [nh, N, d_v] or None (zero).  Returns float64 dict(dv [nh,T,d_v], dalpha [nh,T],
    dbeta [nh,T], dsc_w [nh,T,W], dsc_r [nh,T,R], dM0 [nh,N,d_v]) (dM0 per (sequence,
    head): a learned M_0 shared by the batch receives the sum over the batch).
    """
    M = _c(M_init, np.float64)
    nh, N, dv = M.shape
    iw, sw = _c(idx_w, np.int32), _c(sc_w, np.float32)
    ir, sr = _c(idx_r, np.int32), _c(sc_r, np.float32)
    vv = _c(v, np.float32)
    a, b = _c(alpha, np.float32), _c(beta, np.float32)
    T, W = iw.shape[1], iw.shape[2]
    R = ir.shape[2]
    dO = _c(dO, np.float64)
    G = np.zeros((nh, N, dv), np.float64) if dMT is None else np.array(dMT, np.float64, order="C", copy=True)
    out = dict(dv=np.empty((nh, T, dv)), dalpha=np.empty((nh, T)), dbeta=np.empty((nh, T)),
               dsc_w=np.empty((nh, T, W)), dsc_r=np.empty((nh, T, R)))
    rc = _load().oracle_scan_backward(M.ctypes.data, nh, N, dv, T, W, R, iw.ctypes.data, sw.ctypes.data,
                                      ir.ctypes.data, sr.ctypes.data, vv.ctypes.data, a.ctypes.data,
                                      b.ctypes.data, dO.ctypes.data, G.ctypes.data, out["dv"].ctypes.data,
                                      out["dalpha"].ctypes.data, out["dbeta"].ctypes.data,
                                      out["dsc_w"].ctypes.data, out["dsc_r"].ctypes.data, _threads(n_threads))
    if rc != 0:
        raise ValueError("oracle_scan_backward: bad sizes or slot index out of range")
    out["dM0"] = G
    return out


def select_backward(S: int, idx, dsc):
    """Gradient of the selected scores with respect to the two halves they are sums of:
    sc = half0[flat // S] + half1[flat % S], so each half entry receives the sum of dsc
    over the selected slots that use it.  idx: int [..., K]; dsc: [..., K].
    Returns float64 [..., 2, S]."""
    idx = np.asarray(idx)
    dsc = np.asarray(dsc, np.float64)
    lead = idx.shape[:-1]
    flat_i = idx.reshape(-1, idx.shape[-1])
    flat_d = dsc.reshape(-1, dsc.shape[-1])
    out = np.zeros((flat_i.shape[0], 2, S))
    rows = np.arange(flat_i.shape[0])[:, None]
    np.add.at(out[:, 0], (rows, flat_i // S), flat_d)
    np.add.at(out[:, 1], (rows, flat_i % S), flat_d)
    return out.reshape(lead + (2, S))


def project(x, w, H: int, S: int):
    """The key and query projections ("Meccanismo Core" item 2: k' and q' are projections of
    the token features whose two halves are the sub-scores; "Design IsoFLOP": plain linear
    layers).  x: [..., D] (any float values, e.g. bf16 patterns decoded to fp32);
    w: [4*H*S, D], one row per output column: k' columns in (head, half, index) order,
    then q' columns in the same order.

    Returns float64 (kp, qp, mag), each [lead..., H, 2, S] when x is [lead..., D] with the
    token axis moved behind the head axis for x of shape [B, T, D] (kp[b, h, t, half, s]);
    mag = sum_d |x_d w_nd| per output (the scale of the accumulation's rounding error).
    The products and sums are exact up to fp64 rounding (one library matmul)."""
    x64 = np.asarray(x, np.float64)
    w64 = np.asarray(w, np.float64)
    if w64.shape != (4 * H * S, x64.shape[-1]):
        raise ValueError("w must be [4*H*S, D]")
    y = x64 @ w64.T                                   # [..., 4HS]
    mag = np.abs(x64) @ np.abs(w64).T
    lead = x64.shape[:-1]

    def split(a):
        a = a.reshape(lead + (2, H, 2, S))            # (k' or q', head, half, index)
        a = np.moveaxis(a, len(lead), 0)              # [2, lead..., H, 2, S]
        if len(lead) == 2:                            # [B, T, ...] -> [B, H, T, 2, S]
            a = np.moveaxis(a, 3, 2)
        return a[0], a[1]

    kp, qp = split(y)
    mk, mq = split(mag)
    return kp, qp, (mk, mq)
