"""Thin Python binding of the SDM C ABI (include/sdm.h) for torch tensors.

Argument marshalling only: every step of the path runs in libsdm.so's CUDA
kernels.  There is no CPU fallback: if the library is missing and cannot be built,
or a tensor is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import functools
import math
import os
import sys
import threading

import torch

from . import build as _build

SDM_F32, SDM_BF16 = 0, 1
SDM_DEV_INDEX_RANGE, SDM_DEV_DUP_WRITE, SDM_DEV_TIMEOUT = 1, 2, 4
SDM_MAX_S, SDM_MAX_K = 4096, 1024

_lock = threading.Lock()
_lib = None


class SDMError(RuntimeError):
    """A non-zero status returned by the SDM C ABI."""

    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {lib().sdm_status_str(status).decode()} (status {status})")


def lib() -> ctypes.CDLL:
    """The loaded libsdm.so (built in-tree on first use if absent or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(path)
            p, i, ll, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_size_t
            ull, f = ctypes.c_ulonglong, ctypes.c_float
            L.sdm_status_str.argtypes = [i]
            L.sdm_status_str.restype = ctypes.c_char_p
            L.sdm_init_state_from_M0.argtypes = [p, p, i, i, ll, i, p]
            L.sdm_select.argtypes = [p, p, i, i, i, i, i, i, i, p, p, p, p, p]
            L.sdm_select_tuned.argtypes = [p, p, i, i, i, i, i, i, i, p, p, p, p, i, p]
            L.sdm_scan_workspace_size.argtypes = [i, i, i, i, i, i]
            L.sdm_scan_workspace_size.restype = sz
            L.sdm_scan_forward.argtypes = [p, p, p, p, p, p, i, p, p, i, i, i, ll, i, i, i, p, p, sz, p, p]
            L.sdm_scan_forward_tuned.argtypes = [p, p, p, p, p, p, i, p, p, i, i, i, ll, i, i, i, p, p, sz,
                                                 p, i, i, p, p, p]
            L.sdm_scan_launch_info.argtypes = [i, i, i, i, i, p, p, p, p]
            L.sdm_gen_inputs.argtypes = [ull, i, i, i, i, i, ll, i, i, i, f, i, p, p, p, p, p, p, p]
            L.sdm_gen_M0.argtypes = [ull, i, ll, i, f, p, p]
            L.sdm_forward_workspace_size.argtypes = [i, i, i, i, i, i, i]
            L.sdm_forward_workspace_size.restype = sz
            L.sdm_forward_chunks.argtypes = [i, i]
            L.sdm_forward_tuned.argtypes = [p, p, i, p, i, p, p, p, p, i, i, i, i, i, i, i, p, p, p, p, p, p,
                                            sz, p, i, p, p]
            L.sdm_forward.argtypes = [p, p, i, p, i, p, p, p, p, i, i, i, i, i, i, i, p, p, p, p, p, p, sz, p, p]
            L.sdm_forward_streamed.argtypes = [p, p, i, p, i, p, p, p, p, i, i, i, i, i, i, i, p, p, p, p, p,
                                               p, sz, p, i, p, p, p]
            L.sdm_copy_rows_async.argtypes = [p, sz, p, sz, sz, sz, p]
            L.sdm_scan_forward_train.argtypes = [p, p, p, p, p, p, i, p, p, i, i, i, ll, i, i, i, p, p, p, p, sz, p, p]
            L.sdm_scan_backward_workspace_size.argtypes = [i, i, i, i, i, i]
            L.sdm_scan_backward_workspace_size.restype = sz
            L.sdm_scan_backward.argtypes = [p, p, p, p, p, i, p, p, p, p, p, i, i, i, ll, i, i, i, p, p, p, p, p, p,
                                            p, p, sz, p]
            L.sdm_scan_backward_workspace_size_ex.argtypes = [i, i, i, ll, i, i, i, ctypes.c_uint]
            L.sdm_scan_backward_workspace_size_ex.restype = sz
            L.sdm_scan_backward_ex.argtypes = [p, p, p, p, p, i, p, p, p, p, p, i, i, i, ll, i, i, i, p, p, p, p,
                                               p, p, p, ctypes.c_uint, p, sz, p]
            L.sdm_select_backward.argtypes = [p, p, i, i, i, i, i, p, p]
            L.sdm_decode_step.argtypes = [p, p, i, p, i, p, p, p, i, i, i, i, i, i, p, p, p, p, p, p, p]
            L.sdm_decode_step_supported.argtypes = [i, i, i, i, i, i, i]
            L.sdm_decode_table_words.argtypes = [i, i, i]
            L.sdm_decode_table.argtypes = [p, i, i, i, p]
            L.sdm_decode_step_tabled.argtypes = [p, p, i, p, i, p, p, p, i, i, i, i, i, i, p, p, p, p, p, p, p, p]
            L.sdm_project_kq_tuned.argtypes = [p, p, i, i, i, i, i, p, p, p, i, i, p]
            L.sdm_test_bounded_wait.argtypes = [i, ull, p, p, p]
            L.sdm_test_project_stall.argtypes = [p, p, i, i, i, i, i, p, p, i, i, i, ull, p, p]
            L.sdm_fill_state.argtypes = [p, f, i, i, ll, i, p]
            L.sdm_project_select_workspace_size.argtypes = [i, i, i, i, i, i]
            L.sdm_project_select_workspace_size.restype = sz
            L.sdm_project_select.argtypes = [p, p, i, i, i, i, i, i, i, p, p, p, p, p, sz, p, p]
            for name in ("sdm_init_state_from_M0", "sdm_select", "sdm_select_tuned", "sdm_scan_forward",
                         "sdm_scan_forward_tuned", "sdm_scan_launch_info", "sdm_gen_inputs", "sdm_gen_M0",
                         "sdm_forward_chunks", "sdm_forward_tuned", "sdm_forward", "sdm_scan_forward_train",
                         "sdm_scan_backward", "sdm_scan_backward_ex", "sdm_select_backward", "sdm_project_select",
                         "sdm_fill_state", "sdm_test_project_stall", "sdm_decode_table_words",
                         "sdm_decode_table", "sdm_decode_step_tabled"):
                getattr(L, name).restype = i
            _lib = L
    return _lib


def library_path() -> str:
    return _build.LIB


def _first_cuda_tensor(values):
    for a in values:
        if isinstance(a, torch.Tensor):
            if a.is_cuda:
                return a
        elif isinstance(a, (tuple, list)):
            t = _first_cuda_tensor(a)
            if t is not None:
                return t
        elif isinstance(a, dict):
            t = _first_cuda_tensor(a.values())
            if t is not None:
                return t
    return None


def _on_tensor_device(fn):
    """Runs fn with the device of its first CUDA tensor argument current, so the library
    (which launches on the current device and looks up per-device state there) works on
    the tensors' GPU whatever device the caller had current.  _need then rejects tensors
    of one call that sit on different devices."""
    @functools.wraps(fn)
    def wrapped(*args, **kwargs):
        t = _first_cuda_tensor(list(args) + list(kwargs.values()))
        if t is None:
            return fn(*args, **kwargs)
        with torch.cuda.device(t.device):
            return fn(*args, **kwargs)
    return wrapped


def _call(fn: str, *args):
    st = getattr(lib(), fn)(*args)
    if st != 0:
        raise SDMError(fn, st)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SDM_F32
    if t.dtype == torch.bfloat16:
        return SDM_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _need(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, but the call runs on cuda:{torch.cuda.current_device()}: "
                         "every tensor of one call must be on the same device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


@_on_tensor_device
def init_state_from_M0(M: torch.Tensor, M0: torch.Tensor) -> torch.Tensor:
    """M[b, h] = M0[h] for every b.  M: fp32 [B, H, N, d_v]; M0: fp32 [H, N, d_v]."""
    _need(M, "M", torch.float32)
    B, H, N, dv = M.shape
    _need(M0, "M0", torch.float32, (H, N, dv))
    _call("sdm_init_state_from_M0", _p(M), _p(M0), B, H, N, dv, _stream(M.device))
    return M


@_on_tensor_device
def fill_state(M: torch.Tensor, value: float = 0.0) -> torch.Tensor:
    """Every entry of M (fp32 [B, H, N, d_v]) set to value, e.g. the backward pass's adjoint
    table cleared when the final state carries no gradient."""
    _need(M, "M", torch.float32)
    B, H, N, dv = M.shape
    _call("sdm_fill_state", _p(M), ctypes.c_float(value), B, H, N, dv, _stream(M.device))
    return M


SELECT_AUTO, SELECT_GENERAL, SELECT_COUNTING = 0, 1, 2


@_on_tensor_device
def select(kp: torch.Tensor, qp: torch.Tensor, W: int, R: int, out=None, path: int = SELECT_AUTO):
    """Top-W slots of k' and top-R slots of q' for every (b, h, t).

    kp, qp: [B, H, T, 2, S] fp32 or bf16.  Returns (idx_w int32 [B,H,T,W], sc_w fp32,
    idx_r int32 [B,H,T,R], sc_r fp32), best first.  path: SELECT_AUTO, or force the
    general or the counting kernel (the same results, bit for bit)."""
    _need(kp, "kp")
    B, H, T, two, S = kp.shape
    if two != 2:
        raise ValueError("kp must be [B, H, T, 2, S]")
    _need(qp, "qp", kp.dtype, kp.shape)
    if out is None:
        dev = kp.device
        out = (torch.empty((B, H, T, W), dtype=torch.int32, device=dev),
               torch.empty((B, H, T, W), dtype=torch.float32, device=dev),
               torch.empty((B, H, T, R), dtype=torch.int32, device=dev),
               torch.empty((B, H, T, R), dtype=torch.float32, device=dev))
    idx_w, sc_w, idx_r, sc_r = out
    _need(idx_w, "idx_w", torch.int32, (B, H, T, W))
    _need(sc_w, "sc_w", torch.float32, (B, H, T, W))
    _need(idx_r, "idx_r", torch.int32, (B, H, T, R))
    _need(sc_r, "sc_r", torch.float32, (B, H, T, R))
    _call("sdm_select_tuned", _p(kp), _p(qp), _dtype_code(kp), B, H, T, S, W, R, _p(idx_w), _p(sc_w),
          _p(idx_r), _p(sc_r), int(path), _stream(kp.device))
    return idx_w, sc_w, idx_r, sc_r


def scan_workspace_size(B: int, H: int, T: int, d_v: int, W: int, R: int) -> int:
    return int(lib().sdm_scan_workspace_size(B, H, T, d_v, W, R))


def scan_workspace(B, H, T, d_v, W, R, device) -> torch.Tensor:
    """A device buffer large enough for scan_forward on these sizes."""
    return torch.empty(max(16, scan_workspace_size(B, H, T, d_v, W, R)), dtype=torch.uint8, device=device)


@_on_tensor_device
def scan_forward(M, idx_w, sc_w, idx_r, sc_r, v, alpha, beta, o=None, workspace=None,
                 dev_err=None, cols_per_cta: int = 0, prefetch_depth: int = 0, event_after_plan=None,
                 wait_before_scan=None):
    """Sparse gated-delta scan over T tokens, continuing from the state in M (updated in
    place).  M: fp32 [B,H,N,d_v]; idx/sc from select; v: [B,H,T,d_v] fp32/bf16;
    alpha, beta: fp32 [B,H,T].  Returns o fp32 [B,H,T,d_v].  event_after_plan: optional
    torch.cuda.Event recorded between the planning kernel and the scan kernel;
    wait_before_scan: optional torch.cuda.Event the scan kernel (but not the planning
    kernel, which does not read M) waits for."""
    _need(M, "M", torch.float32)
    B, H, N, dv = M.shape
    _need(idx_w, "idx_w", torch.int32)
    T, W = idx_w.shape[2], idx_w.shape[3]
    _need(idx_w, "idx_w", torch.int32, (B, H, T, W))
    _need(sc_w, "sc_w", torch.float32, (B, H, T, W))
    R = idx_r.shape[3]
    _need(idx_r, "idx_r", torch.int32, (B, H, T, R))
    _need(sc_r, "sc_r", torch.float32, (B, H, T, R))
    _need(v, "v", None, (B, H, T, dv))
    _need(alpha, "alpha", torch.float32, (B, H, T))
    _need(beta, "beta", torch.float32, (B, H, T))
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=torch.float32, device=M.device)
    _need(o, "o", torch.float32, (B, H, T, dv))
    if workspace is None:
        workspace = scan_workspace(B, H, T, dv, W, R, M.device)
    _need(workspace, "workspace", torch.uint8)
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32)
    if event_after_plan is not None and event_after_plan.cuda_event == 0:
        event_after_plan.record()  # torch creates its events lazily; the library records it again
    if wait_before_scan is not None and wait_before_scan.cuda_event == 0:
        raise ValueError("wait_before_scan must have been recorded")
    _call("sdm_scan_forward_tuned", _p(M), _p(idx_w), _p(sc_w), _p(idx_r), _p(sc_r), _p(v),
          _dtype_code(v), _p(alpha), _p(beta), B, H, T, N, dv, W, R, _p(o), _p(workspace),
          workspace.numel(), _p(dev_err), int(cols_per_cta), int(prefetch_depth),
          None if event_after_plan is None else ctypes.c_void_p(event_after_plan.cuda_event),
          None if wait_before_scan is None else ctypes.c_void_p(wait_before_scan.cuda_event),
          _stream(M.device))
    return o


NOALLOC_SCRATCH_BYTES = 64 << 20


@_on_tensor_device
def scan_forward_noalloc(M, idx_w, sc_w, idx_r, sc_r, v, alpha, beta, o, dev_err=None):
    """scan_forward for callers that cannot allocate device memory where the scan runs.

    Same inputs and results as scan_forward, but the library uses its own fixed device
    scratch (NOALLOC_SCRATCH_BYTES, held on every GPU that loads the library) instead of a
    workspace, and the output buffer o must be passed in: nothing is allocated here or in
    the library.  Sizes whose workspace would exceed the scratch raise SDMError.  Calls
    share the scratch, so they must not overlap on the GPU (keep them on one stream); the
    first call on a device should come before any stream capture."""
    L = lib()
    f = L.sdm_scan_forward_noalloc
    p, i, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
    f.argtypes = [p, p, p, p, p, p, i, p, p, i, i, i, ll, i, i, i, p, p, p]
    f.restype = i
    _need(M, "M", torch.float32)
    B, H, N, dv = M.shape
    T, W, R = idx_w.shape[2], idx_w.shape[3], idx_r.shape[3]
    _need(idx_w, "idx_w", torch.int32, (B, H, T, W))
    _need(sc_w, "sc_w", torch.float32, (B, H, T, W))
    _need(idx_r, "idx_r", torch.int32, (B, H, T, R))
    _need(sc_r, "sc_r", torch.float32, (B, H, T, R))
    _need(v, "v", None, (B, H, T, dv))
    _need(alpha, "alpha", torch.float32, (B, H, T))
    _need(beta, "beta", torch.float32, (B, H, T))
    _need(o, "o", torch.float32, (B, H, T, dv))
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32)
    st = f(_p(M), _p(idx_w), _p(sc_w), _p(idx_r), _p(sc_r), _p(v), _dtype_code(v), _p(alpha), _p(beta),
           B, H, T, N, dv, W, R, _p(o), _p(dev_err), _stream(M.device))
    if st != 0:
        raise SDMError("sdm_scan_forward_noalloc", st)
    return o


def scan_launch_info(B: int, H: int, d_v: int, W: int, R: int) -> dict:
    vals = [ctypes.c_int(0) for _ in range(4)]
    _call("sdm_scan_launch_info", B, H, d_v, W, R, *[ctypes.byref(x) for x in vals])
    return dict(cols_per_cta=vals[0].value, prefetch_depth=vals[1].value, blocks=vals[2].value,
                smem_bytes=vals[3].value)


@_on_tensor_device
def gen_inputs(seed: int, B: int, H: int, T: int, S: int, d_v: int, in_dtype: torch.dtype,
               alpha_lo: float, beta_kind: int, half_bias=None, b_off: int = 0, t_off: int = 0,
               T_total=None, device="cuda", out=None):
    """Synthetic inputs drawn on the device (bit-identical to the host generator).

    Returns dict(kp, qp [B,H,T,2,S], v [B,H,T,d_v] in_dtype, alpha, beta fp32 [B,H,T])."""
    T_total = T if T_total is None else T_total
    if out is None:
        out = dict(kp=torch.empty((B, H, T, 2, S), dtype=in_dtype, device=device),
                   qp=torch.empty((B, H, T, 2, S), dtype=in_dtype, device=device),
                   v=torch.empty((B, H, T, d_v), dtype=in_dtype, device=device),
                   alpha=torch.empty((B, H, T), dtype=torch.float32, device=device),
                   beta=torch.empty((B, H, T), dtype=torch.float32, device=device))
    dev = next(t for t in out.values() if t is not None).device
    with torch.cuda.device(dev):
        for k in ("kp", "qp", "v", "alpha", "beta"):
            if out.get(k) is not None:
                _need(out[k], k)
        if half_bias is not None:
            _need(half_bias, "half_bias", torch.float32, (S,))
        _call("sdm_gen_inputs", ctypes.c_ulonglong(seed), B, H, T, b_off, t_off, T_total, S, d_v,
              SDM_BF16 if in_dtype == torch.bfloat16 else SDM_F32,
              ctypes.c_float(alpha_lo), int(beta_kind), _p(half_bias), _p(out.get("kp")), _p(out.get("qp")),
              _p(out.get("v")), _p(out.get("alpha")), _p(out.get("beta")), _stream(dev))
    return out


@_on_tensor_device
def gen_M0(seed: int, H: int, N: int, d_v: int, scale: float = 0.02, device="cuda", out=None):
    """Synthetic learned initial state M0 = scale * N(0, 1), fp32 [H, N, d_v]."""
    if out is None:
        out = torch.empty((H, N, d_v), dtype=torch.float32, device=device)
    with torch.cuda.device(out.device):
        _need(out, "M0", torch.float32, (H, N, d_v))
        _call("sdm_gen_M0", ctypes.c_ulonglong(seed), H, N, d_v, ctypes.c_float(scale), _p(out),
              _stream(out.device))
    return out


_side_streams = {}


def side_stream(device) -> torch.cuda.Stream:
    """A second stream per device, used to overlap the state initialisation (HBM writes)
    with the selection (compare/select work); created once.  It has high priority: the
    selection kernel queues many short blocks, and without priority the initialisation's
    blocks would only get SM slots once that queue drained."""
    dev = torch.device(device)
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    if key not in _side_streams:
        _side_streams[key] = torch.cuda.Stream(device=key, priority=-1)
    return _side_streams[key]


def forward_chunks(T: int, chunks: int = 0) -> int:
    """Token chunks forward() pipelines T tokens in (chunks=0: the automatic choice)."""
    return lib().sdm_forward_chunks(T, chunks)


def forward_workspace(B: int, H: int, T: int, d_v: int, W: int, R: int, device, chunks: int = 0) -> torch.Tensor:
    n = lib().sdm_forward_workspace_size(B, H, T, d_v, W, R, chunks)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


@_on_tensor_device
def forward(kp, qp, v, alpha, beta, M0, W: int, R: int, M=None, workspace=None, dev_err=None,
            overlap: bool = True, out=None, o=None, chunks: int = 0, scan_events=None,
            input_events=None):
    """One SDM forward pass over a batch: state from M0 (or, with M0=None, from the state
    already in M), selection, scan.  Returns (o, M, (idx_w, sc_w, idx_r, sc_r)).

    overlap=True runs sdm_forward: the selection of token chunk c+1 overlaps the scan of
    chunk c on the library's own streams (chunks=0: automatic).  overlap=False runs the
    three steps one after the other on the current stream.  Both give the same bits.
    scan_events: optional list of 2 * forward_chunks(T, chunks) torch.cuda.Event, recorded
    around each chunk's scan kernel.  input_events: optional list of forward_chunks(T, chunks)
    torch.cuda.Event (or None entries), already recorded: chunk c's selection and planning
    wait for input_events[c] (sdm_forward_streamed), e.g. its token window's copy
    (copy_token_window); the state initialisation does not wait."""
    B, H, T, _, S = kp.shape
    dv = v.shape[-1]
    if M is None:
        if M0 is None:
            raise ValueError("M0=None continues from M, which must then be given")
        M = torch.empty((B, H, S * S, dv), dtype=torch.float32, device=kp.device)
    if not overlap:
        if M0 is not None:
            init_state_from_M0(M, M0)
        sel = select(kp, qp, W, R, out=out)
        o = scan_forward(M, *sel, v, alpha, beta, o=o, workspace=workspace, dev_err=dev_err)
        return o, M, sel
    _need(kp, "kp")
    _need(qp, "qp", kp.dtype, tuple(kp.shape))
    _need(M, "M", torch.float32, (B, H, S * S, dv))
    if M0 is not None:
        _need(M0, "M0", torch.float32, (H, S * S, dv))
    _need(v, "v", None, (B, H, T, dv))
    _need(alpha, "alpha", torch.float32, (B, H, T))
    _need(beta, "beta", torch.float32, (B, H, T))
    if out is None:
        dev = kp.device
        out = (torch.empty((B, H, T, W), dtype=torch.int32, device=dev), torch.empty((B, H, T, W), device=dev),
               torch.empty((B, H, T, R), dtype=torch.int32, device=dev), torch.empty((B, H, T, R), device=dev))
    idx_w, sc_w, idx_r, sc_r = out
    _need(idx_w, "idx_w", torch.int32, (B, H, T, W))
    _need(sc_w, "sc_w", torch.float32, (B, H, T, W))
    _need(idx_r, "idx_r", torch.int32, (B, H, T, R))
    _need(sc_r, "sc_r", torch.float32, (B, H, T, R))
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=torch.float32, device=M.device)
    _need(o, "o", torch.float32, (B, H, T, dv))
    if workspace is None:
        workspace = forward_workspace(B, H, T, dv, W, R, M.device, chunks)
    _need(workspace, "workspace", torch.uint8)
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32)
    ev_arr = None
    if scan_events is not None:
        if len(scan_events) != 2 * forward_chunks(T, chunks):
            raise ValueError("scan_events needs 2 * forward_chunks(T, chunks) events")
        for e in scan_events:
            if e.cuda_event == 0:
                e.record()  # torch creates its events lazily; the library records it again
        ev_arr = (ctypes.c_void_p * len(scan_events))(*[e.cuda_event for e in scan_events])
    in_arr = None
    if input_events is not None:
        if not overlap:
            raise ValueError("input_events needs the pipelined pass (overlap=True)")
        if len(input_events) != forward_chunks(T, chunks):
            raise ValueError("input_events needs forward_chunks(T, chunks) events")
        in_arr = (ctypes.c_void_p * len(input_events))(
            *[None if e is None or e.cuda_event == 0 else e.cuda_event for e in input_events])
    _call("sdm_forward_streamed", _p(kp), _p(qp), _dtype_code(kp), _p(v), _dtype_code(v), _p(alpha),
          _p(beta), _p(M0), _p(M), B, H, T, S, dv, W, R, _p(idx_w), _p(sc_w), _p(idx_r), _p(sc_r), _p(o),
          _p(workspace), workspace.numel(), _p(dev_err), int(chunks), ev_arr, in_arr, _stream(M.device))
    return o, M, out


def _huge_page_bytes() -> int:
    """The size of a transparent huge page on this host (2 MB with 4 KB base pages, 512 MB
    with 64 KB ones); 2 MB where the kernel does not say."""
    try:
        with open("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size") as f:
            n = int(f.read().strip())
        return n if n > 0 and n & (n - 1) == 0 else 1 << 21
    except (OSError, ValueError):
        return 1 << 21


def pinned_empty(shape, dtype, device=None) -> torch.Tensor:
    """Page-locked host memory for staging copies to and from the GPU (copy_token_window,
    Tensor.copy_).  The pages are asked for as transparent huge pages where the OS allows,
    then registered with CUDA: the copy engines then need few address translations, which
    keeps host-device copies at full rate while the GPU is busy even when the host's memory is
    fragmented (small pinned pages there slowed a streamed loop's copies several-fold).  Falls
    back to torch's pinned allocator where that is not possible.  The registration and the
    mapping go with the last reference to the buffer (after the device has finished its
    work, so a copy still in flight never meets unlocked pages)."""
    import mmap
    import weakref

    import numpy as np

    shape = tuple(int(x) for x in shape)
    nbytes = int(np.prod(shape, dtype=np.int64)) * torch.empty((), dtype=dtype).element_size()
    madv = getattr(mmap, "MADV_HUGEPAGE", None)
    huge = _huge_page_bytes()
    # A huge page covers only a whole, aligned stretch of the mapping, so the buffer starts on
    # a huge-page boundary and its pages are whole huge pages; buffers under a quarter of one
    # (where that rounding would waste most of the page) take torch's pinned allocator.
    if nbytes < huge // 4 or madv is None or not hasattr(mmap, "MAP_ANONYMOUS"):
        return torch.empty(shape, dtype=dtype, pin_memory=True)
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    size = (nbytes + huge - 1) // huge * huge + huge  # room to start on a huge-page boundary
    mm = mmap.mmap(-1, size, flags=mmap.MAP_PRIVATE | mmap.MAP_ANONYMOUS)
    try:
        mm.madvise(madv)
    except OSError:
        pass
    raw = np.frombuffer(mm, dtype=np.uint8)
    skip = (-raw.ctypes.data) % huge
    buf = raw[skip:skip + nbytes]
    span = (nbytes + huge - 1) // huge * huge
    raw[skip:skip + span] = 0  # fault whole huge pages in
    if sys.platform.startswith("linux"):
        try:  # MADV_COLLAPSE: put what did not come as huge pages onto huge pages, before locking
            mm.madvise(25, skip, span)
        except (OSError, ValueError):
            pass
    with torch.cuda.device(dev):
        rc = int(torch.cuda.cudart().cudaHostRegister(buf.ctypes.data, nbytes, 0))
    if rc != 0:
        del buf, raw
        mm.close()
        return torch.empty(shape, dtype=dtype, pin_memory=True)
    ptr = buf.ctypes.data

    def release(ptr=ptr, mm=mm, dev=dev):
        with torch.cuda.device(dev):
            # copies still in flight from or to these pages finish before they are unlocked
            torch.cuda.synchronize(dev)
            torch.cuda.cudart().cudaHostUnregister(ptr)

    fin = weakref.finalize(buf, release)  # buf lives as long as the tensor's storage
    fin.atexit = False  # at interpreter exit the process teardown releases it
    return torch.from_numpy(buf).view(dtype).view(shape)


def copy_token_window(dst, src, t0: int, t1: int, stream=None):
    """Copy tokens t0 .. t1-1 of every (b, h) from src to dst, both [B, H, T, ...] contiguous
    with the same shape and dtype, one on the GPU and the other pinned host memory (or both on
    the GPU): one strided copy of B*H rows (sdm_copy_rows_async) on `stream` (default: the
    current stream of the GPU tensor's device)."""
    if dst.shape != src.shape or dst.dtype != src.dtype:
        raise ValueError("dst and src must have the same shape and dtype")
    if not (dst.is_contiguous() and src.is_contiguous()):
        raise ValueError("dst and src must be contiguous")
    if dst.dim() < 3 or not 0 <= t0 <= t1 <= dst.shape[2]:
        raise ValueError("need [B, H, T, ...] tensors and 0 <= t0 <= t1 <= T")
    if not (dst.is_cuda or src.is_cuda):
        raise ValueError("one side must be on the GPU")
    for t in (dst, src):
        if not t.is_cuda and not t.is_pinned():
            raise ValueError("host tensors must be pinned")
    dev = dst.device if dst.is_cuda else src.device
    tok = dst.element_size() * math.prod(dst.shape[3:])  # bytes of one token of one (b, h)
    pitch = tok * dst.shape[2]
    off = tok * t0
    s = torch.cuda.current_stream(dev) if stream is None else stream
    _call("sdm_copy_rows_async", ctypes.c_void_p(dst.data_ptr() + off), pitch, ctypes.c_void_p(src.data_ptr() + off),
          pitch, tok * (t1 - t0), dst.shape[0] * dst.shape[1], ctypes.c_void_p(s.cuda_stream))


@_on_tensor_device
def scan_forward_train(M, idx_w, sc_w, idx_r, sc_r, v, alpha, beta, o=None, workspace=None, dev_err=None):
    """scan_forward that also keeps what scan_backward needs.  Returns (o, w_prev, r_rows):
    w_prev [B,H,T,W,d_v] every write row before its update, r_rows [B,H,T,R,d_v] every read
    row as read (fp32)."""
    _need(M, "M", torch.float32)
    B, H, N, dv = M.shape
    T, W, R = idx_w.shape[2], idx_w.shape[3], idx_r.shape[3]
    for t_, n_, dt_, sh_ in ((idx_w, "idx_w", torch.int32, (B, H, T, W)), (sc_w, "sc_w", torch.float32, (B, H, T, W)),
                             (idx_r, "idx_r", torch.int32, (B, H, T, R)), (sc_r, "sc_r", torch.float32, (B, H, T, R)),
                             (v, "v", None, (B, H, T, dv)), (alpha, "alpha", torch.float32, (B, H, T)),
                             (beta, "beta", torch.float32, (B, H, T))):
        _need(t_, n_, dt_, sh_)
    if o is None:
        o = torch.empty((B, H, T, dv), dtype=torch.float32, device=M.device)
    w_prev = torch.empty((B, H, T, W, dv), dtype=torch.float32, device=M.device)
    r_rows = torch.empty((B, H, T, R, dv), dtype=torch.float32, device=M.device)
    if workspace is None:
        workspace = scan_workspace(B, H, T, dv, W, R, M.device)
    _call("sdm_scan_forward_train", _p(M), _p(idx_w), _p(sc_w), _p(idx_r), _p(sc_r), _p(v), _dtype_code(v),
          _p(alpha), _p(beta), B, H, T, N, dv, W, R, _p(o), _p(w_prev), _p(r_rows), _p(workspace),
          workspace.numel(), _p(dev_err), _stream(M.device))
    return o, w_prev, r_rows


BWD_FINAL_ZERO = 1  # sdm_scan_backward_ex flag: dL/dM_T = 0, G's entry contents ignored
BWD_DM0_ONLY = 2    # with BWD_FINAL_ZERO: dM0 wanted, G per (b, h) not (unread rows left as they were)


def backward_workspace_size(B: int, H: int, T: int, N: int, d_v: int, W: int, R: int,
                            final_zero: bool = False) -> int:
    """Bytes of workspace scan_backward needs (sdm_scan_backward_workspace_size_ex)."""
    return int(lib().sdm_scan_backward_workspace_size_ex(B, H, T, N, d_v, W, R,
                                                         BWD_FINAL_ZERO if final_zero else 0))


@_on_tensor_device
def scan_backward(idx_w, sc_w, idx_r, sc_r, v, alpha, beta, w_prev, r_rows, dO, G, shared_M0: bool = True,
                  workspace=None, final_zero: bool = False, dm0_only: bool = False):
    """Reverse-mode pass of the scan for L = sum_t <dO_t, o_t> + <dM_T, M_T>, slots fixed.
    G: fp32 [B,H,N,d_v], in dL/dM_T, out dL/dM_0 per (b, h) (in place).  final_zero: dM_T
    is zero and G's entry contents are ignored (it need not be cleared; the pass skips the
    adjoint rows it knows to be zero).  dm0_only (with final_zero and shared_M0): only the
    batch's dM0 is wanted, so the rows of G no slot reads are not zeroed (G unspecified on
    exit).  Returns dict(dv, dalpha, dbeta, dsc_w, dsc_r, dM0) with dM0 = sum of G over the
    batch (shared_M0) or None."""
    _need(G, "G", torch.float32)
    B, H, N, dv = G.shape
    T, W, R = idx_w.shape[2], idx_w.shape[3], idx_r.shape[3]
    _need(dO, "dO", torch.float32, (B, H, T, dv))
    _need(w_prev, "w_prev", torch.float32, (B, H, T, W, dv))
    _need(r_rows, "r_rows", torch.float32, (B, H, T, R, dv))
    dev = G.device
    out = dict(dv=torch.empty((B, H, T, dv), device=dev), dalpha=torch.empty((B, H, T), device=dev),
               dbeta=torch.empty((B, H, T), device=dev), dsc_w=torch.empty((B, H, T, W), device=dev),
               dsc_r=torch.empty((B, H, T, R), device=dev),
               dM0=torch.empty((H, N, dv), device=dev) if shared_M0 else None)
    if workspace is None:
        n = backward_workspace_size(B, H, T, N, dv, W, R, final_zero)
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
    _call("sdm_scan_backward_ex", _p(idx_w), _p(sc_w), _p(idx_r), _p(sc_r), _p(v), _dtype_code(v), _p(alpha),
          _p(beta), _p(w_prev), _p(r_rows), _p(dO), B, H, T, N, dv, W, R, _p(G), _p(out["dv"]), _p(out["dalpha"]),
          _p(out["dbeta"]), _p(out["dsc_w"]), _p(out["dsc_r"]), _p(out["dM0"]),
          (BWD_FINAL_ZERO if final_zero else 0) | (BWD_DM0_ONLY if dm0_only else 0), _p(workspace),
          workspace.numel(), _stream(dev))
    return out


@_on_tensor_device
def select_backward(idx, dsc, S: int, out=None):
    """Gradient of the selected scores with respect to the halves: [B,H,T,2,S] fp32."""
    _need(idx, "idx", torch.int32)
    B, H, T, K = idx.shape
    _need(dsc, "dsc", torch.float32, (B, H, T, K))
    if out is None:
        out = torch.empty((B, H, T, 2, S), dtype=torch.float32, device=idx.device)
    _call("sdm_select_backward", _p(idx), _p(dsc), B, H, T, S, K, _p(out), _stream(idx.device))
    return out


@_on_tensor_device
def project_kq(x, w, H: int, S: int, out=None, dev_err=None, max_ctas: int = 0, pair: int = -1):
    """The projections x -> k', q' on the tensor cores: one bf16 GEMM, fp32 accumulation,
    outputs rounded to bf16 in the [B, H, T, 2, S] layout ``select`` reads.

    x: [B, T, D] bf16; w: [4*H*S, D] bf16, one row per output column: the k' columns in
    (head, half, index) order, then the q' columns.  max_ctas caps the blocks (0: one per
    SM); pair 2/0/-1: two-SM MMA tiles / single blocks / auto (2 unless there is a single
    row tile).
    Returns (kp, qp)."""
    _need(x, "x", torch.bfloat16)
    if x.dim() != 3:
        raise ValueError("x must be [B, T, D]")
    B, T, D = x.shape
    _need(w, "w", torch.bfloat16, (4 * H * S, D))
    if out is None:
        out = (torch.empty((B, H, T, 2, S), dtype=torch.bfloat16, device=x.device),
               torch.empty((B, H, T, 2, S), dtype=torch.bfloat16, device=x.device))
    kp, qp = out
    _need(kp, "kp", torch.bfloat16, (B, H, T, 2, S))
    _need(qp, "qp", torch.bfloat16, (B, H, T, 2, S))
    _call("sdm_project_kq_tuned", _p(x), _p(w), B, T, D, H, S, _p(kp), _p(qp),
          _p(dev_err) if dev_err is not None else None, int(max_ctas), int(pair), _stream(x.device))
    return kp, qp


def project_select_workspace(B: int, T: int, H: int, S: int, W: int, R: int, device) -> torch.Tensor:
    n = lib().sdm_project_select_workspace_size(B, T, H, S, W, R)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


@_on_tensor_device
def project_select(x, w, H: int, S: int, W: int, R: int, out=None, workspace=None, dev_err=None):
    """The projections x -> k', q' fused with the selection: the top-W slots of k' and the
    top-R slots of q' for every (b, h, t), as select(*project_kq(x, w, H, S), W, R) gives them,
    without k' and q' in device memory.  x: [B, T, D] bf16; w: [4*H*S, D] bf16.
    Returns (idx_w, sc_w, idx_r, sc_r)."""
    _need(x, "x", torch.bfloat16)
    if x.dim() != 3:
        raise ValueError("x must be [B, T, D]")
    B, T, D = x.shape
    _need(w, "w", torch.bfloat16, (4 * H * S, D))
    dev = x.device
    if out is None:
        out = (torch.empty((B, H, T, W), dtype=torch.int32, device=dev),
               torch.empty((B, H, T, W), dtype=torch.float32, device=dev),
               torch.empty((B, H, T, R), dtype=torch.int32, device=dev),
               torch.empty((B, H, T, R), dtype=torch.float32, device=dev))
    idx_w, sc_w, idx_r, sc_r = out
    _need(idx_w, "idx_w", torch.int32, (B, H, T, W))
    _need(sc_w, "sc_w", torch.float32, (B, H, T, W))
    _need(idx_r, "idx_r", torch.int32, (B, H, T, R))
    _need(sc_r, "sc_r", torch.float32, (B, H, T, R))
    if workspace is None:
        workspace = project_select_workspace(B, T, H, S, W, R, dev)
    _need(workspace, "workspace", torch.uint8)
    if dev_err is not None:
        _need(dev_err, "dev_err", torch.int32)
    _call("sdm_project_select", _p(x), _p(w), B, T, D, H, S, W, R, _p(idx_w), _p(sc_w), _p(idx_r), _p(sc_r),
          _p(workspace), workspace.numel(), _p(dev_err), _stream(dev))
    return idx_w, sc_w, idx_r, sc_r


def bounded_wait_check(mode: int, limit_ns: int, device="cuda"):
    """Runs one bounded mbarrier wait of the projection kernel's kind on one warp (mode 0: a
    phase nothing completes, 1: a completed phase, 2: the stop flag already raised) and
    returns (dev_err, elapsed_ns): the error word it reported (SDM_DEV_TIMEOUT when the wait
    gave up) and the wait's duration on the global timer.  Synchronises the device."""
    dev_err = torch.zeros(1, dtype=torch.int32, device=device)
    elapsed = torch.zeros(1, dtype=torch.int64, device=device)
    with torch.cuda.device(dev_err.device):
        _call("sdm_test_bounded_wait", int(mode), ctypes.c_ulonglong(limit_ns), _p(dev_err), _p(elapsed),
              _stream(dev_err.device))
    torch.cuda.synchronize(dev_err.device)
    return int(dev_err.item()), int(elapsed.item())


@_on_tensor_device
def project_stall_check(x, w, H: int, S: int, pair: int, stall_cta: int, stall_step: int, wait_ns: int):
    """The projection kernel with the copy-issuing thread of cluster rank `stall_cta` stopping
    after `stall_step` K steps and every wait limited to wait_ns (sdm_test_project_stall):
    the kernel must stop, drain its copies and report.  Returns the error word (the
    SDM_DEV_TIMEOUT bit set when it stopped).  Synchronises the device."""
    _need(x, "x", torch.bfloat16)
    _need(w, "w", torch.bfloat16)
    B, T, D = x.shape
    kp = torch.empty((B, H, T, 2, S), dtype=torch.bfloat16, device=x.device)
    qp = torch.empty_like(kp)
    dev_err = torch.zeros(1, dtype=torch.int32, device=x.device)
    _call("sdm_test_project_stall", _p(x), _p(w), B, T, D, H, S, _p(kp), _p(qp), int(pair), int(stall_cta),
          int(stall_step), ctypes.c_ulonglong(wait_ns), _p(dev_err), _stream(x.device))
    torch.cuda.synchronize(x.device)
    return int(dev_err.item())


def decode_table(W: int, R: int, S: int, device="cuda") -> torch.Tensor:
    """The staircase table of a (W, R, S) decode step (int32 words on `device`), built once
    by sdm_decode_table; decode_step(table=...) then reads it instead of building it."""
    n = lib().sdm_decode_table_words(W, R, S)
    if n < 0:
        raise ValueError("sizes not supported by the decode step")
    dev = torch.device(device)
    t = torch.empty(n, dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        _call("sdm_decode_table", _p(t), W, R, S, _stream(dev))
    return t


@_on_tensor_device
def decode_step(kp, qp, v, alpha, beta, M, W: int, R: int, out=None, o=None, dev_err=None, table=None):
    """One decode token (T = 1) for every (b, h) in a single kernel: selection, planning and
    the gated write and read on M (in place).  kp, qp [B, H, 1, 2, S]; v [B, H, 1, d_v];
    alpha, beta [B, H, 1]; M [B, H, S*S, d_v] fp32.  Returns (o, (idx_w, sc_w, idx_r, sc_r)),
    bit-identical to select() followed by scan_forward() on the same token.  table: the
    step's staircase table from decode_table(W, R, S) (optional; the same bits)."""
    _need(kp, "kp")
    B, H, T, two, S = kp.shape
    if T != 1 or two != 2:
        raise ValueError("kp must be [B, H, 1, 2, S]")
    _need(qp, "qp", kp.dtype, tuple(kp.shape))
    dv = v.shape[-1]
    _need(v, "v", None, (B, H, 1, dv))
    _need(alpha, "alpha", torch.float32, (B, H, 1))
    _need(beta, "beta", torch.float32, (B, H, 1))
    _need(M, "M", torch.float32, (B, H, S * S, dv))
    if out is None:
        dev = kp.device
        out = (torch.empty((B, H, 1, W), dtype=torch.int32, device=dev), torch.empty((B, H, 1, W), device=dev),
               torch.empty((B, H, 1, R), dtype=torch.int32, device=dev), torch.empty((B, H, 1, R), device=dev))
    if o is None:
        o = torch.empty((B, H, 1, dv), dtype=torch.float32, device=M.device)
    _need(o, "o", torch.float32, (B, H, 1, dv))
    if table is not None:
        n = lib().sdm_decode_table_words(W, R, S)
        _need(table, "table", torch.int32, (n,))
    _call("sdm_decode_step_tabled", _p(kp), _p(qp), _dtype_code(kp), _p(v), _dtype_code(v), _p(alpha),
          _p(beta), _p(M), B, H, S, dv, W, R, _p(out[0]), _p(out[1]), _p(out[2]), _p(out[3]), _p(o),
          _p(dev_err) if dev_err is not None else None, _p(table) if table is not None else None,
          _stream(M.device))
    return o, out


class DecodeStep:
    """One-token decode step for a batch of sequences with resident state, captured once
    into a CUDA graph and replayed per token: the single-kernel decode_step (fused=True, the
    default where its shared memory fits), else the selection, planning and scan kernels.

    The state M [B, H, N, d_v] stays in place across steps; each step takes k', q' halves
    [B, H, 1, 2, S], v [B, H, 1, d_v] and alpha, beta [B, H, 1] and returns o [B, H, 1, d_v]
    (the step's static output buffer: copy it before the next step if it must be kept).
    With the single kernel, inputs laid out as the static buffers (contiguous, same dtypes,
    on M's device) are read where they are: one launch, no copy.  Otherwise they are copied
    into the static buffers and the graph (or the unfused kernels) runs on those.  Chaining
    steps gives exactly the result of one scan over the same tokens."""

    def __init__(self, M, W: int, R: int, in_dtype=torch.bfloat16, S=None, fused=None):
        B, H, N, dv = M.shape
        S = int(round(N ** 0.5)) if S is None else S
        if fused is None:
            code = SDM_BF16 if in_dtype == torch.bfloat16 else SDM_F32
            with torch.cuda.device(M.device):
                fused = lib().sdm_decode_step_supported(code, B, H, S, dv, W, R) == 0
        self.fused = bool(fused)
        if S * S != N:
            raise ValueError("N must be a square")
        dev = M.device
        self.M, self.W, self.R = M, W, R
        self.kp = torch.zeros((B, H, 1, 2, S), dtype=in_dtype, device=dev)
        self.qp = torch.zeros_like(self.kp)
        self.v = torch.zeros((B, H, 1, dv), dtype=in_dtype, device=dev)
        self.alpha = torch.ones((B, H, 1), dtype=torch.float32, device=dev)
        self.beta = torch.zeros((B, H, 1), dtype=torch.float32, device=dev)
        self.sel = (torch.empty((B, H, 1, W), dtype=torch.int32, device=dev),
                    torch.empty((B, H, 1, W), dtype=torch.float32, device=dev),
                    torch.empty((B, H, 1, R), dtype=torch.int32, device=dev),
                    torch.empty((B, H, 1, R), dtype=torch.float32, device=dev))
        self.o = torch.empty((B, H, 1, dv), dtype=torch.float32, device=dev)
        self.ws = scan_workspace(B, H, 1, dv, W, R, dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        # the staircase table of this shape, built once for every step
        self.table = decode_table(W, R, S, dev) if self.fused else None
        self.graph = None
        # Fixed arguments of the single-kernel launch on the caller's tensors (plain integer
        # addresses: ctypes converts them for the c_void_p parameters).
        self._fn = lib().sdm_decode_step_tabled
        self._codes = (_dtype_code(self.kp), _dtype_code(self.v))
        self._tail = (M.data_ptr(), B, H, S, dv, W, R) + tuple(t.data_ptr() for t in self.sel) + (
            self.o.data_ptr(), self.err.data_ptr(), self.table.data_ptr() if self.fused else None)
        self._bufs = (self.kp, self.qp, self.v, self.alpha, self.beta)
        # what a caller's input must match to be read in place (checked cheaply per call)
        self._sig = tuple((b.dtype, tuple(b.shape)) for b in self._bufs)
        self._dev_index = dev.index
        self._raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)

    def _body(self):
        if self.fused:
            decode_step(self.kp, self.qp, self.v, self.alpha, self.beta, self.M, self.W, self.R,
                        out=self.sel, o=self.o, dev_err=self.err, table=self.table)
            return
        select(self.kp, self.qp, self.W, self.R, out=self.sel)
        scan_forward(self.M, *self.sel, self.v, self.alpha, self.beta, o=self.o, workspace=self.ws,
                     dev_err=self.err)

    def capture(self):
        """Capture the step (selection, planning, scan) into a CUDA graph.  Beforehand the
        same kernels run once on a small dummy problem with the same (B, H, d_v, W, R), so
        that they are loaded and configured outside the capture; the real state is not
        touched until the graph is replayed."""
        B, H, N, dv = self.M.shape
        dev = self.M.device
        s = 1
        while s * s < max(self.W, self.R):
            s += 1
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            kp = torch.zeros((B, H, 1, 2, s), dtype=self.kp.dtype, device=dev)
            sel = select(kp, kp, self.W, self.R)
            Md = torch.zeros((B, H, s * s, dv), dtype=torch.float32, device=dev)
            scan_forward(Md, *sel, self.v, self.alpha, self.beta)
            if self.fused:
                decode_step(kp, kp, self.v, self.alpha, self.beta, Md, self.W, self.R)
        torch.cuda.current_stream(dev).wait_stream(side)
        torch.cuda.synchronize(dev)
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self._body()
        return self

    @property
    def inputs(self) -> dict:
        """The step's static input buffers (kp, qp, v, alpha, beta): a producer that writes
        a token's inputs here directly can then call run() without any copy."""
        return dict(kp=self.kp, qp=self.qp, v=self.v, alpha=self.alpha, beta=self.beta)

    def run(self):
        """One step on the inputs already in the static buffers; returns o (static)."""
        if self.graph is None:
            self._body()
        else:
            self.graph.replay()
        return self.o

    def _direct(self, kp, qp, v, alpha, beta) -> bool:
        """The single kernel launched on the caller's tensors where they are laid out as the
        static buffers (no copy); False where they are not."""
        if not self.fused:
            return False
        idx = self._dev_index
        for x, (dt, shape) in zip((kp, qp, v, alpha, beta), self._sig):
            if (not isinstance(x, torch.Tensor) or x.dtype is not dt or x.shape != shape
                    or x.get_device() != idx or not x.is_contiguous()):
                return False
        if torch.cuda.current_device() != idx:
            with torch.cuda.device(self.M.device):
                return self._direct(kp, qp, v, alpha, beta)
        stream = (self._raw_stream(idx) if self._raw_stream is not None
                  else torch.cuda.current_stream(self.M.device).cuda_stream)
        st = self._fn(kp.data_ptr(), qp.data_ptr(), self._codes[0], v.data_ptr(), self._codes[1],
                      alpha.data_ptr(), beta.data_ptr(), *self._tail, stream)
        if st != 0:
            raise SDMError("sdm_decode_step_tabled", st)
        return True

    def __call__(self, kp, qp, v, alpha, beta):
        if self._direct(kp, qp, v, alpha, beta):
            return self.o
        self.kp.copy_(kp, non_blocking=True)
        self.qp.copy_(qp, non_blocking=True)
        self.v.copy_(v, non_blocking=True)
        self.alpha.copy_(alpha, non_blocking=True)
        self.beta.copy_(beta, non_blocking=True)
        if self.graph is None:
            self._body()
        else:
            self.graph.replay()
        return self.o
