"""sdm_scan_forward_noalloc: the scan for callers that cannot allocate device memory
where they run it (a serving loop that forbids allocation on its request path, or a
host program that owns no allocator and passes only its own buffers).  It uses the
library's fixed device scratch instead of a caller workspace.

Called here through the C ABI directly and checked against sdm_scan_forward (which
takes a workspace) on the same inputs, twice in a row with problems of different
sizes, so that the second call also shows that what the first one left in the shared
scratch does not leak into its result.  Kept in its own file that pytest collects
last.
"""
import ctypes

import numpy as np
import pytest
import torch

import sparse_state_linear_sdm_gb300 as sdm

pytestmark = pytest.mark.gpu

TOL = 2e-4           # max |x - x_ref| <= TOL * (1 + |x_ref|), as in the other parity tests
SDM_ESCRATCH = -8
SCRATCH_BYTES = 64 << 20


def _entry():
    f = sdm.lib().sdm_scan_forward_noalloc
    p, i, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
    f.argtypes = [p, p, p, p, p, p, i, p, p, i, i, i, ll, i, i, i, p, p, p]
    f.restype = i
    return f


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _problem(seed, B, H, T, S, dv, W, R):
    g = torch.Generator(device="cuda").manual_seed(seed)
    kp = torch.randn((B, H, T, 2, S), generator=g, device="cuda").to(torch.bfloat16)
    qp = torch.randn((B, H, T, 2, S), generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn((B, H, T, dv), generator=g, device="cuda").to(torch.bfloat16)
    alpha = 0.9 + 0.1 * torch.rand((B, H, T), generator=g, device="cuda")
    beta = torch.rand((B, H, T), generator=g, device="cuda")
    M0 = 0.02 * torch.randn((H, S * S, dv), generator=g, device="cuda")
    sel = sdm.select(kp, qp, W, R)
    return sel, v, alpha, beta, M0


def _scaled_err(got, want):
    g = got.double().cpu().numpy()
    w = want.double().cpu().numpy()
    return float((np.abs(g - w) / (1.0 + np.abs(w))).max())


@pytest.mark.parametrize("first,second", [((2, 3, 300, 16, 32, 12, 10), (1, 2, 97, 8, 16, 5, 7))])
def test_noalloc_matches_workspace_scan_on_two_calls(first, second):
    f = _entry()
    for k, (B, H, T, S, dv, W, R) in enumerate((first, second)):
        sel, v, alpha, beta, M0 = _problem(100 + k, B, H, T, S, dv, W, R)
        N = S * S
        M_ref = M0[None].repeat(B, 1, 1, 1)   # copies (an expand of size-1 dims would alias M0)
        o_ref = sdm.scan_forward(M_ref, *sel, v, alpha, beta)
        M = M0[None].repeat(B, 1, 1, 1)
        o = torch.full((B, H, T, dv), float("nan"), device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        st = f(_ptr(M), *[_ptr(x) for x in sel], _ptr(v), 1, _ptr(alpha), _ptr(beta), B, H, T, N, dv, W, R,
               _ptr(o), _ptr(err), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, sdm.lib().sdm_status_str(st)
        torch.cuda.synchronize()
        assert err.item() == 0
        assert _scaled_err(o, o_ref) <= TOL, f"call {k}: outputs differ"
        assert _scaled_err(M, M_ref) <= TOL, f"call {k}: final state differs"


def test_noalloc_refuses_problems_beyond_its_scratch():
    f = _entry()
    fake = ctypes.c_void_p(0x10000)  # never touched: every check runs on the host first
    B, H, T, dv, W, R = 8, 8, 512, 128, 128, 128
    need = sdm.scan_workspace_size(B, H, T, dv, W, R)
    assert need > SCRATCH_BYTES
    st = f(fake, fake, fake, fake, fake, fake, 1, fake, fake, B, H, T, 1 << 20, dv, W, R, fake, None, None)
    assert st == SDM_ESCRATCH
    assert b"no-allocation scratch" in sdm.lib().sdm_status_str(st)


def test_noalloc_python_wrapper_matches_workspace_scan():
    """The binding's scan_forward_noalloc (argument checks, the device made current for
    the call) gives the workspace scan's results on two calls in a row."""
    for k, (B, H, T, S, dv, W, R) in enumerate(((1, 2, 150, 16, 16, 6, 9), (2, 1, 40, 8, 32, 4, 4))):
        sel, v, alpha, beta, M0 = _problem(200 + k, B, H, T, S, dv, W, R)
        M_ref = M0[None].repeat(B, 1, 1, 1)
        o_ref = sdm.scan_forward(M_ref, *sel, v, alpha, beta)
        M = M0[None].repeat(B, 1, 1, 1)
        o = torch.full((B, H, T, dv), float("nan"), device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        sdm.scan_forward_noalloc(M, *sel, v, alpha, beta, o, dev_err=err)
        torch.cuda.synchronize()
        assert err.item() == 0
        assert _scaled_err(o, o_ref) <= TOL, f"call {k}: outputs differ"
        assert _scaled_err(M, M_ref) <= TOL, f"call {k}: final state differs"
