"""Host logic of bench.py that needs no GPU: the algorithmic bytes per head-token, the
whole-job rate, the clock summary, the peak lookup, the workload choice, and the gating
of the committed ncu records (DRAM traffic, instruction counts) by kernel source hash,
workload and launch shape."""
import hashlib
import json
import types

import pytest

import bench
from sparse_state_linear_sdm_gb300 import workloads as wl


def test_scan_bytes_per_head_token():
    # W rows gathered and scattered, R rows gathered (fp32, d_v each), v (bf16), alpha and
    # beta (fp32), o (fp32): (2*128 + 128)*128*4 + 128*2 + 8 + 128*4
    assert bench.scan_bytes_per_head_token(wl.B16H4_T8192) == 197_384
    # fp32 v on the tiny workload: (2*8 + 8)*16*4 + 16*4 + 8 + 16*4
    assert bench.scan_bytes_per_head_token(wl.TINY_F32) == 1_672


def test_zero_adjoint_slots_brute_force():
    """The zero-adjoint slot counts behind the backward's roofline bytes, against a brute
    force over every slot: a write slot at t is zero when no read at t' >= t selects its
    row, a read slot when no read at t' > t does."""
    import numpy as np
    import torch
    rng = np.random.default_rng(5)
    B, H, T, W, R, N = 2, 3, 30, 4, 5, 24
    iw = rng.integers(0, N, (B, H, T, W)).astype(np.int32)
    ir = np.stack([[[rng.choice(N, R, replace=False) for _ in range(T)] for _ in range(H)] for _ in range(B)])
    ir = ir.astype(np.int32)
    sel = (torch.from_numpy(iw), None, torch.from_numpy(ir), None)
    zw = zr = 0
    for b in range(B):
        for h in range(H):
            for t in range(T):
                zw += sum(all(x not in ir[b, h, u] for u in range(t, T)) for x in iw[b, h, t])
                zr += sum(all(x not in ir[b, h, u] for u in range(t + 1, T)) for x in ir[b, h, t])
    assert bench.zero_adjoint_slots(sel, N, torch) == (zw, zr)
    assert 0 < zw < B * H * T * W and 0 < zr < B * H * T * R


def test_whole_job_rate_counts_every_rank_over_the_slowest_time():
    # 2 ranks x 1000 units x 5 steps in 250 ms
    assert bench.whole_job_rate(1000, 5, 2, 250.0) == pytest.approx(40_000.0)


def _sampler_with_rows(tmp_path, rows):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc = object()          # as if nvidia-smi had been started
    s.out = open(tmp_path / "clocks.csv", "w+")
    s.out.write("".join(r + "\n" for r in rows))
    return s


def test_clock_summary_median_max_and_reasons(tmp_path):
    rows = [
        "0, 2070, 2070, 950.1, 0x0, Not Active, Not Active, Not Active, Not Active",
        "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
        "0, 2010, 2070, 1201.5, 0x0, Not Active, Not Active, Not Active, Not Active",
        "garbage line",
        "0, [N/A], 2070, 1000, 0x0, Not Active, Not Active, Not Active, Not Active",
    ]
    got = _sampler_with_rows(tmp_path, rows).summary()
    assert got == {"sm_mhz": 2010.0, "sm_max_mhz": 2070.0, "samples": 3, "reasons": ["sw_power_cap"]}


def test_clock_summary_reports_thermal_and_hw_slowdowns(tmp_path):
    rows = ["0, 1500, 2070, 1400, 0x68, Active, Active, Active, Not Active"]
    got = _sampler_with_rows(tmp_path, rows).summary()
    assert got["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_sampler_is_none():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc = None
    assert s.summary() is None


def test_hbm_peak_measured_or_fallback(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.hbm_peak() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6698.5}))
    assert bench.hbm_peak() == (6698.5, "measured")


def _args(**kw):
    base = dict(config="3", seed=None, override="")
    base.update(kw)
    return types.SimpleNamespace(**base)


def test_workload_by_position_name_seed_and_override():
    assert bench.workload(_args()) == wl.B16H4_T8192
    assert bench.workload(_args(config="B4H8-T2048-N65536-dv64-W32")) == wl.B4H8_T2048
    c = bench.workload(_args(config="1", seed=11))
    assert c.seed == 11 and c.name.endswith("(seed 11)") and c.T == wl.B4H8_T2048.T
    c = bench.workload(_args(override="S=256,T=512"))
    assert (c.S, c.T, c.B) == (256, 512, wl.B16H4_T8192.B)
    with pytest.raises(KeyError):
        bench.workload(_args(config="no-such-workload"))


def _sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def test_scan_traffic_record_is_used_only_for_its_kernel_source(tmp_path, monkeypatch):
    rec = {"dram_bytes_per_head_token": 200_000.0, "source_sha256": _sha(bench.SCAN_SRC)}
    path = tmp_path / "scan.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(path))
    assert bench.traffic_per_launch(32_768) == pytest.approx(200_000.0 * 32_768)
    rec["source_sha256"] = "0" * 64
    path.write_text(json.dumps(rec))
    assert bench.traffic_per_launch(32_768) is None
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(tmp_path / "absent.json"))
    assert bench.traffic_per_launch(32_768) is None


def test_projection_traffic_record_gated_by_shape_and_launch(tmp_path, monkeypatch):
    rec = {"gemm": [131072, 16384, 2048], "dram_bytes_per_launch": 9.5e9,
           "source_sha256": _sha(bench.PROJECT_SRC)}
    path = tmp_path / "proj.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "PROJECT_TRAFFIC_FILE", str(path))
    default = types.SimpleNamespace(max_ctas=0, pair=-1)
    assert bench.project_traffic([131072, 16384, 2048], default) == 9.5e9
    assert bench.project_traffic([16384, 16384, 2048], default) is None
    assert bench.project_traffic([131072, 16384, 2048], types.SimpleNamespace(max_ctas=0, pair=0)) is None
    assert bench.project_traffic([131072, 16384, 2048], types.SimpleNamespace(max_ctas=76, pair=-1)) is None
    rec["source_sha256"] = "0" * 64
    path.write_text(json.dumps(rec))
    assert bench.project_traffic([131072, 16384, 2048], default) is None


def test_select_roofline_from_the_instruction_record(tmp_path, monkeypatch):
    h = hashlib.sha256()
    for p in bench.SELECT_SRC:
        with open(p, "rb") as f:
            h.update(f.read())
    assert h.hexdigest() == bench.select_source_sha()
    cfg = wl.B16H4_T8192
    rec = {"warp_instructions_per_selection": 10_000.0, "shape": [cfg.S, cfg.W, cfg.R, cfg.in_dtype],
           "source_sha256": h.hexdigest()}
    path = tmp_path / "sel.json"
    path.write_text(json.dumps(rec))
    monkeypatch.setattr(bench, "SELECT_FILE", str(path))
    units = cfg.head_tokens
    got = bench.select_roofline(cfg, units, 12.0, {"sm_mhz": 2000.0})
    # two selections (write and read) per head-token
    assert got["achieved"] == pytest.approx(10_000.0 * 2 * units / 12e-3 / 1e9)
    assert got["peak"] == pytest.approx(152 * 4 * 2000.0 / 1e3)
    assert got["frac"] == pytest.approx(got["achieved"] / got["peak"])
    assert got["bound"] == "alu"
    # another shape, or another source, has no record; the stream workload shares the shape
    assert bench.select_roofline(wl.B4H8_T2048, units, 12.0, None) is None
    assert bench.select_roofline(wl.STREAM_B1H4_T1M, units, 12.0, None) is not None
    rec["source_sha256"] = "0" * 64
    path.write_text(json.dumps(rec))
    assert bench.select_roofline(cfg, units, 12.0, None) is None

