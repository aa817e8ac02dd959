"""C ABI checks that need no GPU: the library builds and loads, exports every
function include/sdm.h declares, and rejects bad arguments on the host before
launching anything."""
import ctypes
import os
import re
import subprocess

import pytest

import sparse_state_linear_sdm_gb300 as sdm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdm.h")

EINVAL, EALIGN, EUNSUPPORTED, ENOSPACE = -1, -2, -6, -7


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\**\s+\**(sdm_[A-Za-z_0-9]+)\s*\(", text, re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("sdm_init_state_from_M0", "sdm_select", "sdm_scan_forward", "sdm_scan_workspace_size",
              "sdm_status_str"):
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = sdm.lib()
    out = subprocess.run(["nm", "-D", "--defined-only", sdm.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT\s+(sdm_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_status_strings():
    lib = sdm.lib()
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert lib.sdm_status_str(code)
    assert lib.sdm_status_str(-6) == b"sizes beyond the library's limits"


FAKE = ctypes.c_void_p(0x10000)      # 16-byte aligned, never dereferenced on these paths
ODD = ctypes.c_void_p(0x10004)


def test_select_rejects_bad_arguments_without_launching():
    lib = sdm.lib()
    args = lambda **kw: dict(dict(kp=FAKE, qp=FAKE, dt=1, B=1, H=1, T=4, S=8, W=4, R=4), **kw)

    def call(a, ptrs=(FAKE, FAKE, FAKE, FAKE)):
        return lib.sdm_select(a["kp"], a["qp"], a["dt"], a["B"], a["H"], a["T"], a["S"], a["W"], a["R"],
                              *ptrs, None)

    assert call(args(S=0)) == EINVAL
    assert call(args(W=0)) == EINVAL
    assert call(args(W=65)) == EINVAL           # W > N = 64
    assert call(args(dt=7)) == EINVAL
    assert call(args(B=0)) == EINVAL
    assert call(args(S=5000, W=4)) == EUNSUPPORTED
    assert call(args(S=64, W=2000)) == EUNSUPPORTED
    assert call(args(kp=ODD)) == EALIGN
    assert call(args(), ptrs=(FAKE, ODD, FAKE, FAKE)) == EALIGN
    assert call(args(T=0)) == 0                 # nothing to do


def test_scan_rejects_bad_arguments_without_launching():
    lib = sdm.lib()

    def call(B=1, H=1, T=8, N=64, dv=16, W=4, R=4, v_dt=0, M=FAKE, ws=FAKE, ws_bytes=1 << 30, cols=0, pd=0):
        return lib.sdm_scan_forward_tuned(M, FAKE, FAKE, FAKE, FAKE, FAKE, v_dt, FAKE, FAKE, B, H, T, N, dv, W,
                                          R, FAKE, ws, ws_bytes, None, cols, pd, None, None, None)

    assert call(dv=6) == EINVAL
    assert call(dv=0) == EINVAL
    assert call(W=65) == EINVAL
    assert call(R=0) == EINVAL
    assert call(v_dt=3) == EINVAL
    assert call(pd=4) == EINVAL
    assert call(W=1025, N=1 << 20) == EUNSUPPORTED
    assert call(M=ODD) == EALIGN
    assert call(ws=ODD) == EALIGN
    assert call(ws_bytes=10) == ENOSPACE
    assert call(T=0) == 0


def test_workspace_size_formula():
    lib = sdm.lib()
    # record = slots (W+R int32) + weights (W+R fp32) + sources (W+R int16) + 16 B gates + d_v fp32
    assert lib.sdm_scan_workspace_size(16, 4, 8192, 128, 128, 128) == 16 * 4 * 8192 * (1024 + 1024 + 512 + 16 + 512)
    assert lib.sdm_scan_workspace_size(1, 1, 64, 16, 8, 8) == 64 * (64 + 64 + 32 + 16 + 64)
    # W + R = 7 pads to 8 int32/fp32 and 8 int16
    assert lib.sdm_scan_workspace_size(1, 1, 1, 4, 3, 4) == 32 + 32 + 16 + 16 + 16
    assert lib.sdm_scan_workspace_size(1, 1, 0, 16, 8, 8) == 0


def test_init_and_gen_reject_bad_arguments():
    lib = sdm.lib()
    assert lib.sdm_init_state_from_M0(FAKE, FAKE, 1, 1, 16, 6, None) == EINVAL
    assert lib.sdm_init_state_from_M0(ODD, FAKE, 1, 1, 16, 8, None) == EALIGN
    assert lib.sdm_gen_inputs(0, 1, 1, 4, 0, 2, 5, 8, 8, 1, ctypes.c_float(0.9), 1, None, None, None, None,
                              None, None, None) == EINVAL   # t_off + T > T_total
    assert lib.sdm_gen_M0(0, 1, 16, 4, ctypes.c_float(0.02), ODD, None) == EALIGN


def test_api_requires_cuda_tensors():
    """Every entry point of the binding refuses host tensors before doing anything: there is
    no CPU path to fall back to."""
    import torch
    B, H, T, S, dv, W, R = 1, 1, 4, 8, 8, 4, 4
    kp = torch.zeros(B, H, T, 2, S)
    v = torch.zeros(B, H, T, dv)
    ab = torch.zeros(B, H, T)
    M = torch.zeros(B, H, S * S, dv)
    M0 = torch.zeros(H, S * S, dv)
    iw = torch.zeros(B, H, T, W, dtype=torch.int32)
    sw = torch.zeros(B, H, T, W)
    calls = [
        lambda: sdm.select(kp, kp, W, R),
        lambda: sdm.init_state_from_M0(M, M0),
        lambda: sdm.scan_forward(M, iw, sw, iw, sw, v, ab, ab),
        lambda: sdm.forward(kp, kp, v, ab, ab, M0, W, R),
        lambda: sdm.forward(kp, kp, v, ab, ab, M0, W, R, overlap=False),
        lambda: sdm.decode_step(kp[:, :, :1], kp[:, :, :1], v[:, :, :1], ab[:, :, :1], ab[:, :, :1], M, W, R),
        lambda: sdm.project_kq(torch.zeros(B, T, 16, dtype=torch.bfloat16),
                               torch.zeros(4 * H * S, 16, dtype=torch.bfloat16), H, S),
        lambda: sdm.select_backward(iw, sw, S),
    ]
    for call in calls:
        with pytest.raises(TypeError, match="must be a CUDA tensor"):
            call()


def test_forward_rejects_bad_arguments_without_launching():
    lib = sdm.lib()

    def call(B=1, H=1, T=8, S=8, dv=16, W=4, R=4, in_dt=1, v_dt=0, ws=FAKE, ws_bytes=1 << 30, chunks=0,
             M0=None, kp=FAKE, M=FAKE):
        return lib.sdm_forward_tuned(kp, FAKE, in_dt, FAKE, v_dt, FAKE, FAKE, M0, M, B, H, T, S, dv, W, R,
                                     FAKE, FAKE, FAKE, FAKE, FAKE, ws, ws_bytes, None, chunks, None, None)

    assert call(dv=6) == EINVAL
    assert call(in_dt=3) == EINVAL
    assert call(v_dt=3) == EINVAL
    assert call(W=65) == EINVAL                 # more slots than N = S * S = 64
    assert call(chunks=-1) == EINVAL
    assert call(S=5000) == EUNSUPPORTED
    assert call(kp=ODD) == EALIGN
    assert call(M=ODD) == EALIGN
    assert call(M0=ODD) == EALIGN
    assert call(ws=ODD) == EALIGN
    assert call(ws_bytes=16) == ENOSPACE
    # the streamed variant checks the same arguments before it looks at its events
    streamed = lib.sdm_forward_streamed(FAKE, FAKE, 1, FAKE, 0, FAKE, FAKE, None, FAKE, 1, 1, 8, 8, 6, 4, 4,
                                        FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1 << 30, None, 0, None, None, None)
    assert streamed == EINVAL                  # d_v = 6


def test_copy_rows_checks_its_arguments_without_copying():
    lib = sdm.lib()
    assert lib.sdm_copy_rows_async(None, 64, FAKE, 64, 64, 2, None) == EINVAL
    assert lib.sdm_copy_rows_async(FAKE, 64, None, 64, 64, 2, None) == EINVAL
    assert lib.sdm_copy_rows_async(FAKE, 32, FAKE, 64, 64, 2, None) == EINVAL   # pitch below the row
    assert lib.sdm_copy_rows_async(FAKE, 64, FAKE, 32, 64, 2, None) == EINVAL
    assert lib.sdm_copy_rows_async(FAKE, 64, FAKE, 64, 64, 0, None) == 0        # nothing to copy
    assert lib.sdm_copy_rows_async(FAKE, 64, FAKE, 64, 0, 2, None) == 0


def test_forward_chunking_and_workspace_sizes():
    lib = sdm.lib()
    assert lib.sdm_forward_chunks(8192, 0) == 8      # 1024 tokens per chunk from T = 8192 on
    assert lib.sdm_forward_chunks(8191, 0) == 16     # about 512 tokens per chunk below
    assert lib.sdm_forward_chunks(65536, 0) == 64
    assert lib.sdm_forward_chunks(8192, 3) == 3
    assert lib.sdm_forward_chunks(1000, 0) == 2
    assert lib.sdm_forward_chunks(500, 0) == 1
    assert lib.sdm_forward_chunks(5, 8) == 5         # never more chunks than tokens
    assert lib.sdm_forward_chunks(0, 0) == 0
    # one record, W = R = 10 (20 slots), d_v = 16: slots, weights, sources (padded to 8),
    # alpha/beta block, v
    rec = 4 * 20 + 4 * 20 + 2 * 24 + 16 + 4 * 16
    assert rec == 288
    # the staircase of the outer top-K: pairs (p, q) of the two inner lists with
    # (p + 1)(q + 1) <= K (sized for inner lists of K entries); one table for W, one for R
    stair = sum(1 for p in range(10) for q in range(10) if (p + 1) * (q + 1) <= 10)
    assert stair == 27
    # two record buffers of B*H*ceil(T/chunks) records, each rounded up to 256 bytes, then
    # both staircases (4 bytes per pair) rounded up to 256 bytes
    assert lib.sdm_forward_workspace_size(2, 3, 100, 16, 10, 10, 4) == \
        2 * ((6 * 25 * rec + 255) // 256 * 256) + (2 * stair * 4 + 255) // 256 * 256
    assert lib.sdm_forward_workspace_size(1, 1, 0, 16, 4, 4, 0) == 0


def test_projection_rejects_bad_arguments_without_launching():
    L = sdm.lib()
    L.sdm_project_kq.argtypes = [ctypes.c_void_p, ctypes.c_void_p] + [ctypes.c_int] * 5 + \
        [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    ok = ctypes.c_void_p(1 << 20)   # never dereferenced: every call below fails its checks
    odd = ctypes.c_void_p((1 << 20) + 8)
    call = lambda x, w, B, T, D, H, S, kp, qp: L.sdm_project_kq(x, w, B, T, D, H, S, kp, qp, None, None)
    assert call(ok, ok, 1, 4, 12, 1, 4, ok, ok) == EINVAL        # D % 8 != 0
    assert call(ok, ok, 1, 4, 0, 1, 4, ok, ok) == EINVAL         # D < 8
    assert call(ok, ok, 0, 4, 64, 1, 4, ok, ok) == EINVAL        # B < 1
    assert call(ok, ok, 1, 4, 64, 1, 0, ok, ok) == EINVAL        # S < 1
    assert call(ok, ok, 1, 4, 64, 1, 5000, ok, ok) == EUNSUPPORTED
    assert call(None, ok, 1, 4, 64, 1, 4, ok, ok) == EALIGN
    assert call(ok, odd, 1, 4, 64, 1, 4, ok, ok) == EALIGN
    assert call(ok, ok, 1, 4, 64, 1, 4, ok, odd) == EALIGN


def test_bounded_wait_check_rejects_bad_arguments_without_launching():
    L = sdm.lib()
    ok = ctypes.c_void_p(1 << 20)   # never dereferenced: every call below fails its checks
    call = lambda mode, limit, err, el=None: L.sdm_test_bounded_wait(mode, limit, err, el, None)
    assert call(3, 1000, ok) == EINVAL                  # unknown mode
    assert call(-1, 1000, ok) == EINVAL
    assert call(0, 10 ** 9 + 1, ok) == EINVAL           # limit above one second
    assert call(0, 1000, None) == EINVAL                # the error word is required
    assert call(0, 1000, ctypes.c_void_p((1 << 20) + 2)) == EALIGN
    assert call(0, 1000, ok, ctypes.c_void_p((1 << 20) + 4)) == EALIGN


def test_backward_flags_and_workspace_sizes():
    """sdm_scan_backward_ex: the zero-final-adjoint flag's workspace (part | last-read table |
    zero bits, each rounded to 16 bytes), unknown flags refused, size checks before launching."""
    lib = sdm.lib()
    B, H, T, N, dv, W, R = 2, 3, 10, 64, 16, 5, 7
    up16 = lambda x: (x + 15) // 16 * 16
    part = B * H * T * 1 * (2 * W + R) * 4            # d_v = 16: one 16-column slice per (b, h)
    wts = B * H * T * (W + R) * 4                     # the softmax weights of every token
    flags = B * H * T * 4 * 4                         # per token: zero bits (W + R), same-token bits (W), padded to 16 B
    base = up16(part) + up16(wts) + up16(flags)
    assert lib.sdm_scan_backward_workspace_size(B, H, T, dv, W, R) == base
    assert lib.sdm_scan_backward_workspace_size_ex(B, H, T, N, dv, W, R, 0) == base
    assert lib.sdm_scan_backward_workspace_size_ex(B, H, T, N, dv, W, R, 1) == base + up16(B * H * N * 4)
    assert lib.sdm_scan_backward_workspace_size_ex(1, 1, 5, 64, 8, 40, 33, 1) == (
        up16(5 * 1 * 113 * 4) + up16(5 * 73 * 4) + up16(5 * 8 * 4) + up16(64 * 4))   # W + R = 73: 3 + 2 words
    assert lib.sdm_scan_backward_workspace_size_ex(B, H, T, N, dv, W, R, 2) == base      # dM0 only: no table
    assert lib.sdm_scan_backward_workspace_size_ex(B, H, T, N, dv, W, R, 3) == base + up16(B * H * N * 4)
    assert lib.sdm_scan_backward_workspace_size_ex(B, H, T, N, dv, W, R, 4) == 0         # unknown bit
    assert lib.sdm_scan_backward_workspace_size_ex(B, H, 0, N, dv, W, R, 1) == up16(B * H * N * 4)

    def call(flags=1, ws=FAKE, ws_bytes=1 << 30, dv_=dv, G=FAKE, dM0=None):
        return lib.sdm_scan_backward_ex(FAKE, FAKE, FAKE, FAKE, FAKE, 0, FAKE, FAKE, FAKE, FAKE, FAKE, B, H, T, N,
                                        dv_, W, R, G, FAKE, FAKE, FAKE, FAKE, FAKE, dM0, flags, ws, ws_bytes, None)

    assert call(flags=2) == EINVAL              # dM0 only without a dM0
    assert call(flags=3) == EINVAL
    assert call(flags=4) == EINVAL              # unknown bit
    assert call(flags=5, dM0=FAKE) == EINVAL
    assert call(flags=3, dM0=FAKE, ws_bytes=base) == ENOSPACE
    assert call(dv_=6) == EINVAL
    assert call(ws=ODD) == EALIGN
    assert call(G=ODD) == EALIGN
    assert call(ws_bytes=base) == ENOSPACE      # the zero flag needs the table


def test_project_stall_rejects_bad_arguments_without_launching():
    lib = sdm.lib()

    def call(B=2, T=300, pair=2, cta=1, step=3, wait=1_000_000, err=FAKE):
        return lib.sdm_test_project_stall(FAKE, FAKE, B, T, 64, 1, 32, FAKE, FAKE, pair, cta, step,
                                          ctypes.c_ulonglong(wait), err, None)

    assert call(pair=1) == EINVAL
    assert call(pair=0, cta=1) == EINVAL
    assert call(cta=2) == EINVAL
    assert call(step=-1) == EINVAL
    assert call(wait=10) == EINVAL
    assert call(wait=2_000_000_000) == EINVAL
    assert call(err=None) == EINVAL
    assert call(B=1, T=100) == EUNSUPPORTED       # one row tile: no pair
    assert call(err=ctypes.c_void_p(0x10002)) == EALIGN   # dev_err is an int


def _stair_words(K, S):
    """Pairs (p, q) of ranks in two sorted lists of min(K, S) keys with (p+1)(q+1) <= K."""
    kin = min(K, S)
    return sum(1 for p in range(kin) for q in range(kin) if (p + 1) * (q + 1) <= K)


def test_decode_table_sizes_and_argument_checks():
    lib = sdm.lib()
    for W, R, S in ((128, 128, 1024), (8, 8, 32), (5, 7, 2), (1, 1, 1), (128, 64, 16), (1024, 3, 4096)):
        assert lib.sdm_decode_table_words(W, R, S) == _stair_words(W, S) + _stair_words(R, S), (W, R, S)
    for W, R, S in ((0, 8, 32), (8, 0, 32), (8, 8, 0), (8, 8, 4097), (1025, 8, 64)):
        assert lib.sdm_decode_table_words(W, R, S) == -1
    assert lib.sdm_decode_table(None, 8, 8, 32, None) == EINVAL
    assert lib.sdm_decode_table(FAKE, 0, 8, 32, None) == EINVAL
    assert lib.sdm_decode_table(ctypes.c_void_p(0x10002), 8, 8, 32, None) == EALIGN
    # a misaligned table is refused before anything else is looked at
    odd_table = ctypes.c_void_p(0x10001)
    assert lib.sdm_decode_step_tabled(FAKE, FAKE, 1, FAKE, 1, FAKE, FAKE, FAKE, 1, 1, 8, 16, 4, 4,
                                      FAKE, FAKE, FAKE, FAKE, FAKE, None, odd_table, None) == EALIGN
    # otherwise the checks of sdm_decode_step apply
    assert lib.sdm_decode_step_tabled(FAKE, FAKE, 1, FAKE, 1, FAKE, FAKE, FAKE, 0, 1, 8, 16, 4, 4,
                                      FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, None) == EINVAL


def test_huge_page_size_is_a_power_of_two():
    from sparse_state_linear_sdm_gb300 import api
    n = api._huge_page_bytes()
    assert n >= 1 << 21 and n & (n - 1) == 0
