#!/usr/bin/env python3
"""SDM forward benchmark: prints one JSON line.

A step is one pass of the whole forward hot path over one batch of synthetic
input resident in HBM: state initialisation from M_0, product-key selection, and
the sparse gated-delta scan (planning kernel + scan kernel).  The default
workload is B=16, H=4, T=8192, N=1,048,576 (S=1024), d_v=128, W=R=128 with bf16
k', q', v and fp32 state (34 GB).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config I] [--seed S] [--impl ours|reference]

With N > 1 (launched by torch.distributed.run) every rank runs its own batch of
sequences (weak scaling; no collective on the data path).  `--impl reference`
times the CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SDM forward head-tokens/s on 1 GB300; achieved HBM GB/s vs roofline"
UNIT = "head-tokens/s"
FALLBACK_HBM_GBS = 6800.0
SCAN_SRC = os.path.join(ROOT, "sparse_state_linear_sdm_gb300", "csrc", "sdm_scan.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "scan_kernel_dram_traffic.json")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="3",
                    help="workload: a name from workloads.CONFIGS or its position (default 3, B16H4-T8192-N1M-dv128-W128)")
    ap.add_argument("--seed", type=int, default=None, help="generator seed (default: the workload's own)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cols", type=int, default=0, help="force scan columns per block (0 = auto)")
    ap.add_argument("--pd", type=int, default=0, help="force scan prefetch depth (0 = auto; one-stream step only)")
    ap.add_argument("--chunks", type=int, default=0, help="token chunks of the pipelined forward (0 = auto)")
    ap.add_argument("--pipeline", choices=["on", "off"], default="on",
                    help="on: sdm_forward (selection of chunk c+1 overlaps the scan of chunk c); "
                         "off: init || select, then plan and scan, one kernel after the other")
    ap.add_argument("--override", default="", help="size overrides for profiling, e.g. S=256,T=512")
    ap.add_argument("--mode", choices=["forward", "decode", "backward", "project"], default="forward",
                    help="decode: one token per step for the batch, state resident, CUDA graph; "
                         "backward: the training backward pass (reverse scan, score and half gradients); "
                         "project: the projections x -> k', q' on the tensor cores")
    ap.add_argument("--dmodel", type=int, default=0, help="feature width D of --mode project (0 = 2048)")
    ap.add_argument("--max-ctas", type=int, default=0, help="blocks of the projection kernel (0 = one per SM)")
    ap.add_argument("--pair", type=int, default=-1, choices=[-1, 0, 2],
                    help="projection kernel: 2 two-SM MMA, 0 single blocks, -1 auto")
    return ap.parse_args()


def workload(args):
    import dataclasses

    from sparse_state_linear_sdm_gb300 import workloads as wl

    cfg = wl.CONFIGS[int(args.config)] if str(args.config).isdigit() else wl.by_name(args.config)
    if args.seed is not None and args.seed != cfg.seed:
        cfg = dataclasses.replace(cfg, name=cfg.name + f" (seed {args.seed})", seed=args.seed)
    if args.override:
        kv = dict(item.split("=") for item in args.override.split(","))
        cfg = dataclasses.replace(cfg, name=cfg.name + f" (sizes overridden: {args.override})",
                                  **{k: int(v) for k, v in kv.items()})
    return cfg


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_batch_offset(rank: int, B: int) -> int:
    """First batch row of this rank: rank r runs sequences r*B .. r*B+B-1 of the logical
    workload (the (b, h) scans are independent, so ranks share nothing)."""
    return rank * B


def max_over_ranks(x: float, device) -> float:
    """Max of a per-rank value over the process group (the slowest rank sets the time)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, steps: int, world: int, max_ms: float) -> float:
    """Head-tokens per second of the whole job: every rank's units over the slowest time."""
    return world * units_per_rank * steps / (max_ms / 1e3)


def scan_bytes_per_head_token(cfg) -> int:
    """Algorithmic HBM bytes of the scan per head-token: W rows gathered and scattered,
    R rows gathered (fp32, d_v each), v, alpha and beta read, o written."""
    elt = 2 if cfg.in_dtype == "bf16" else 4
    return (2 * cfg.W + cfg.R) * cfg.d_v * 4 + cfg.d_v * elt + 8 + cfg.d_v * 4


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


SELECT_SRC = [os.path.join(ROOT, "sparse_state_linear_sdm_gb300", "csrc", f)
              for f in ("sdm_select_impl.cuh", "sdm_select_count.cuh", "sdm_select_bf16.cu",
                        "sdm_select_f32.cu")]
SELECT_FILE = os.path.join(ROOT, "profiles", "select_kernel_instructions.json")
SMS, SMSP_PER_SM = 152, 4


def select_source_sha() -> str:
    h = hashlib.sha256()
    for p in SELECT_SRC:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def select_roofline(cfg, units: int, select_ms: float, clocks):
    """The selection kernel is bound by instruction issue: warp-instructions per selection
    (ncu, a selection of the same S, W, R and input dtype on inputs of the same distribution,
    this kernel source) x selections / its time alone, against one warp-instruction per clock
    per SM sub-partition at the sampled SM clock."""
    try:
        with open(SELECT_FILE) as f:
            rec = json.load(f)
        key = (cfg.S, cfg.W, cfg.R, cfg.in_dtype)
        if rec.get("source_sha256") != select_source_sha() or tuple(rec.get("shape", ())) != key:
            return None
        mhz = (clocks or {}).get("sm_mhz") or 2070.0
        achieved = rec["warp_instructions_per_selection"] * 2 * units / (select_ms / 1e3) / 1e9
        peak = SMS * SMSP_PER_SM * mhz / 1e3
        return {"kernel": "sdm select kernel", "bound": "alu", "achieved": achieved, "peak": peak,
                "unit": "G warp-instructions/s", "frac": achieved / peak,
                "peak_source": f"derived: {SMS} SMs x {SMSP_PER_SM} issue slots/clock x {mhz:.0f} MHz",
                "warp_instructions_per_selection": rec["warp_instructions_per_selection"],
                "ms_alone": select_ms}
    except Exception:
        return None


PROJECT_SRC = os.path.join(ROOT, "sparse_state_linear_sdm_gb300", "csrc", "sdm_project.cu")
PROJECT_TRAFFIC_FILE = os.path.join(ROOT, "profiles", "project_kernel_dram_traffic.json")


def project_traffic(gemm, args):
    """DRAM bytes per projection launch from the committed ncu record, when it was taken on
    this kernel source, this GEMM shape and the default launch shape; else None."""
    try:
        with open(PROJECT_TRAFFIC_FILE) as f:
            rec = json.load(f)
        with open(PROJECT_SRC, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
        if rec.get("source_sha256") != sha or list(rec.get("gemm", [])) != list(gemm):
            return None
        if args.max_ctas != 0 or args.pair != -1:
            return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


def traffic_per_launch(units: int):
    """DRAM bytes per scan launch from the committed ncu summary, scaled from its
    captured case by head-tokens; None if absent or taken on another kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
        with open(SCAN_SRC, "rb") as f:
            sha = hashlib.sha256(f.read()).hexdigest()
        if rec.get("source_sha256") != sha:
            return None
        return float(rec["dram_bytes_per_head_token"]) * units
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock/throttle samples during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return None
        self.out.flush()
        with open(self.out.name) as f:
            rows = [[c.strip() for c in line.split(",")] for line in f if line.strip()]
        os.unlink(self.out.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


def make_state(cfg, rank, dev, torch, sdm, wl):
    """Inputs drawn in HBM by the device generator (rank r draws batch rows
    r*B .. r*B+B-1 of the logical workload) and every buffer of the step."""
    dt = torch.bfloat16 if cfg.in_dtype == "bf16" else torch.float32
    bias = wl.half_bias(cfg)
    bias_d = None if bias is None else torch.from_numpy(bias).to(dev)
    inp = sdm.gen_inputs(cfg.seed, cfg.B, cfg.H, cfg.T, cfg.S, cfg.d_v, dt, cfg.alpha_lo,
                         0 if cfg.beta_kind == "uniform" else 1, half_bias=bias_d,
                         b_off=rank_batch_offset(rank, cfg.B), device=dev)
    st = dict(inp)
    st["M0"] = sdm.gen_M0(cfg.seed, cfg.H, cfg.N, cfg.d_v, float(wl.M0_SCALE), device=dev)
    st["M"] = torch.empty((cfg.B, cfg.H, cfg.N, cfg.d_v), dtype=torch.float32, device=dev)
    sh = (cfg.B, cfg.H, cfg.T)
    st["sel"] = (torch.empty(sh + (cfg.W,), dtype=torch.int32, device=dev),
                 torch.empty(sh + (cfg.W,), dtype=torch.float32, device=dev),
                 torch.empty(sh + (cfg.R,), dtype=torch.int32, device=dev),
                 torch.empty(sh + (cfg.R,), dtype=torch.float32, device=dev))
    st["o"] = torch.empty(sh + (cfg.d_v,), dtype=torch.float32, device=dev)
    st["ws"] = sdm.scan_workspace(cfg.B, cfg.H, cfg.T, cfg.d_v, cfg.W, cfg.R, dev)
    st["fws"] = sdm.forward_workspace(cfg.B, cfg.H, cfg.T, cfg.d_v, cfg.W, cfg.R, dev, 0)
    st["err"] = torch.zeros(1, dtype=torch.int32, device=dev)
    st["side"] = sdm.side_stream(dev)  # high priority: init shares the SMs with the selection
    return st


def run_forward(st, cfg, sdm, args, inp=None, o=None, scan_ev=None, input_ev=None):
    """One forward pass through the public pipelined entry point (sdm_forward): state
    from M0, selection and planning of token chunk c+1 overlapping the scan of chunk c.
    scan_ev: 2 * chunks timing events recorded around each chunk's scan kernel.
    input_ev: chunks events, chunk c's inputs ready (sdm_forward_streamed)."""
    inp = st if inp is None else inp
    o = st["o"] if o is None else o
    if st["fws"].numel() < sdm.lib().sdm_forward_workspace_size(cfg.B, cfg.H, cfg.T, cfg.d_v, cfg.W, cfg.R,
                                                                 args.chunks):
        st["fws"] = sdm.forward_workspace(cfg.B, cfg.H, cfg.T, cfg.d_v, cfg.W, cfg.R, st["M"].device, args.chunks)
    sdm.forward(inp["kp"], inp["qp"], inp["v"], inp["alpha"], inp["beta"], st["M0"], cfg.W, cfg.R, M=st["M"],
                workspace=st["fws"], dev_err=st["err"], out=st["sel"], o=o, chunks=args.chunks,
                scan_events=scan_ev, input_events=input_ev)


def run_step(st, cfg, sdm, args, ev=None, before_select=None, inp=None, o=None):
    """One forward pass: the state initialisation runs on a side stream, overlapped with the
    selection and the planning pass on the main stream; the scan kernel waits for it.
    ev = (start, init end [side], select end, scan start, scan end) CUDA events;
    before_select() enqueues work on the main stream ahead of the selection (the
    end-to-end loop's host->device copies), which then also overlaps the initialisation."""
    import torch

    inp = st if inp is None else inp
    o = st["o"] if o is None else o
    main = torch.cuda.current_stream()
    side = st["side"]
    start = ev[0] if ev else torch.cuda.Event()
    start.record(main)
    side.wait_event(start)
    with torch.cuda.stream(side):
        sdm.init_state_from_M0(st["M"], st["M0"])
    init_done = ev[1] if ev else torch.cuda.Event()
    init_done.record(side)
    if before_select is not None:
        before_select()
    sdm.select(inp["kp"], inp["qp"], cfg.W, cfg.R, out=st["sel"])
    if ev:
        ev[2].record(main)
    sdm.scan_forward(st["M"], *st["sel"], inp["v"], inp["alpha"], inp["beta"], o=o, workspace=st["ws"],
                     dev_err=st["err"], cols_per_cta=args.cols, prefetch_depth=args.pd,
                     event_after_plan=ev[3] if ev else None, wait_before_scan=init_done)
    if ev:
        ev[4].record(main)


ORACLE_SAMPLE_TOKENS = 2048   # tokens of batch row 0 (every head) in one oracle sample
ORACLE_BASELINE_RUNS = 20     # samples timed for cpu_baseline (about 10 s of CPU work)


def cpu_baseline(cfg, wl, oracle, steps=ORACLE_BASELINE_RUNS, tokens=ORACLE_SAMPLE_TOKENS):
    """The oracle, as it stands, on a bounded sample: batch row 0, every head, the first
    `tokens` tokens, fp64 state initialised from M_0 (inside the timed call).  The same
    sample serves cpu_baseline and every step of the reference arm."""
    import numpy as np

    T = min(tokens, cfg.T)
    heads = [(0, h) for h in range(cfg.H)]
    parts = [wl.inputs(cfg, b, b + 1, h, h + 1, 0, T) for b, h in heads]
    host = {k: np.concatenate([p[k].reshape((1,) + p[k].shape[2:]) for p in parts]) for k in parts[0]}
    M0 = wl.initial_state(cfg, 0, cfg.H)
    cores = os.cpu_count() or 1
    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.forward(host["kp"], host["qp"], host["v"], host["alpha"], host["beta"], M0, cfg.W, cfg.R,
                       n_threads=cores)
        times.append(time.perf_counter() - t0)
    units = len(heads) * T
    return dict(value=units * len(times) / sum(times), unit=UNIT, cores=cores, kind="oracle",
                sample=f"{cfg.name}: batch row 0, all {cfg.H} heads, tokens 0..{T - 1} ({units} head-tokens), "
                       f"fp64 state initialised from M_0, selection + scan; {steps} samples, "
                       f"head-tokens over their total time"), times, units


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from sparse_state_linear_sdm_gb300 import workloads as wl

    cfg = workload(args)
    oracle.build()
    base, times, units = cpu_baseline(cfg, wl, oracle, steps=args.warmup + args.steps)
    timed = times[args.warmup:]
    value = units * len(timed) / sum(timed)
    base["value"] = value
    base["sample"] = base["sample"].replace(f"{args.warmup + args.steps} samples", f"one sample per step "
                                            f"({args.warmup} warm-up steps untimed)")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * sum(timed) / len(timed),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_dict(cfg), "cpu_baseline": base,
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


L2_BYTES = 129e6


def l2_note(cfg) -> str:
    """Which of the step's inputs exceed the 129 MB L2 (no flush between timed steps)."""
    elt = 2 if cfg.in_dtype == "bf16" else 4
    parts = {"state table": cfg.B * cfg.H * cfg.N * cfg.d_v * 4,
             "k' and q'": 2 * cfg.B * cfg.H * cfg.T * 2 * cfg.S * elt}
    big = [f"{k} {v / 1e6:.0f} MB" for k, v in parts.items() if v > L2_BYTES]
    small = [f"{k} {v / 1e6:.0f} MB" for k, v in parts.items() if v <= L2_BYTES]
    note = "no L2 flush; larger than the 129 MB L2: " + (", ".join(big) if big else "none")
    return note + ("; within it: " + ", ".join(small) if small else "")


def config_dict(cfg, pipelined=True):
    step = ("sdm_forward: state from M0, then select+plan of token chunk c+1 overlapping the scan of chunk c"
            if pipelined else
            "init_state_from_M0 (side stream) || select, then plan, then scan (waits for init)")
    return {"workload": cfg.name, "B": cfg.B, "H": cfg.H, "T": cfg.T, "N": cfg.N, "d_v": cfg.d_v, "W": cfg.W,
            "R": cfg.R, "inputs": cfg.in_dtype, "state": "f32", "l2": l2_note(cfg), "step": step}


def one_stream_breakdown(st, cfg, sdm, args, torch, dev, reps=3):
    """Each kernel alone, one after the other on the current stream (outside the timed
    region): state initialisation, selection, planning, scan over the whole sequence."""
    E = lambda: torch.cuda.Event(enable_timing=True)
    res = {"init_ms": [], "select_ms": [], "plan_ms": [], "scan_ms": []}
    for r in range(reps + 1):
        e = [E() for _ in range(5)]
        e[0].record()
        sdm.init_state_from_M0(st["M"], st["M0"])
        e[1].record()
        sdm.select(st["kp"], st["qp"], cfg.W, cfg.R, out=st["sel"])
        e[2].record()
        sdm.scan_forward(st["M"], *st["sel"], st["v"], st["alpha"], st["beta"], o=st["o"], workspace=st["ws"],
                         dev_err=st["err"], event_after_plan=e[3])
        e[4].record()
        torch.cuda.synchronize(dev)
        if r == 0:
            continue
        for i, k in enumerate(("init_ms", "select_ms", "plan_ms", "scan_ms")):
            res[k].append(e[i].elapsed_time(e[i + 1]))
    out = {k: sum(v) / len(v) for k, v in res.items()}
    out["sum_ms"] = sum(out.values())
    return out


def run_ours(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import sparse_state_linear_sdm_gb300 as sdm
    from sparse_state_linear_sdm_gb300 import workloads as wl

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = workload(args)
    st = make_state(cfg, rank, dev, torch, sdm, wl)
    torch.cuda.synchronize(dev)

    def barrier():
        if world > 1:
            dist.barrier()

    pipelined = args.pipeline == "on"
    chunks = sdm.forward_chunks(cfg.T, args.chunks) if pipelined else 1
    E = lambda: torch.cuda.Event(enable_timing=True)

    def step(k_ev=None, s_ev=None):
        if pipelined:
            run_forward(st, cfg, sdm, args, scan_ev=s_ev)
        else:
            run_step(st, cfg, sdm, args, k_ev)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if st["err"].item() != 0:
        raise RuntimeError(f"device error flags {st['err'].item()}")

    K = args.steps
    step_ev = [(E(), E()) for _ in range(K)]
    kern_ev = [[E() for _ in range(5)] for _ in range(K)]      # one-stream step: phase events
    scan_ev = [[E() for _ in range(2 * chunks)] for _ in range(K)]  # pipelined step: scan launches
    for group in (step_ev, kern_ev, scan_ev):   # create the events now (torch creates them lazily)
        for e in group:
            for x in e:
                x.record()
    torch.cuda.synchronize(dev)
    barrier()
    torch.cuda.synchronize(dev)
    main = torch.cuda.current_stream(dev)
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for k in range(K):
            step_ev[k][0].record(main)
            step(kern_ev[k], scan_ev[k])
            step_ev[k][1].record(main)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
    barrier()
    total_ms = step_ev[0][0].elapsed_time(step_ev[-1][1])
    total_ms = max_over_ranks(total_ms, dev)
    units_rank = cfg.B * cfg.H * cfg.T
    value = whole_job_rate(units_rank, K, world, total_ms)

    # roofline of the dominant kernel (the scan): its launches, timed by their own events on
    # the stream they run on
    if pipelined:
        launches = [e[2 * c].elapsed_time(e[2 * c + 1]) for e in scan_ev for c in range(chunks)]
        scan_launch_ms = sum(launches) / len(launches)
        units_launch = units_rank / chunks
        phase = {"scan_ms_per_launch": scan_launch_ms, "scan_ms_per_step": scan_launch_ms * chunks,
                 "chunks": chunks, "tokens_per_chunk": -(-cfg.T // chunks),
                 "overlap": "sdm_forward: init (high-priority stream) || staircase table once, then "
                            "select of chunk c+1 (low-priority stream) then its plan (high-priority "
                            "stream) || scan of chunk c (high-priority stream)"}
        phase["alone"] = one_stream_breakdown(st, cfg, sdm, args, torch, dev)
        # init, the staircase table, then select, plan and scan per chunk
        launches_per_step = 2 + 3 * chunks
    else:
        scan_launch_ms = sum(e[3].elapsed_time(e[4]) for e in kern_ev) / K
        units_launch = units_rank
        # init runs on the side stream from the step start; select from the step start on the
        # main stream; plan until the scan starts; scan until the step ends.
        phase = {"init_ms": sum(e[0].elapsed_time(e[1]) for e in kern_ev) / K,
                 "select_ms": sum(e[0].elapsed_time(e[2]) for e in kern_ev) / K,
                 "plan_ms": sum(e[2].elapsed_time(e[3]) for e in kern_ev) / K,
                 "scan_ms": scan_launch_ms,
                 "overlap": "init on a side stream, concurrent with select and plan"}
        launches_per_step = 4
    peak, peak_kind = hbm_peak()
    alg = scan_bytes_per_head_token(cfg) * units_launch
    achieved = alg / (scan_launch_ms / 1e3) / 1e9
    shape = sdm.scan_launch_info(cfg.B, cfg.H, cfg.d_v, cfg.W, cfg.R)
    if not pipelined and (args.cols or args.pd):
        shape["forced"] = {"cols_per_cta": args.cols, "prefetch_depth": args.pd}
    traffic = traffic_per_launch(units_launch)

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": total_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic", "config": config_dict(cfg, pipelined),
            "roofline": {"kernel": "sdm scan kernel", "bound": "hbm", "achieved": achieved, "peak": peak,
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                         else "fallback", "unit": "GB/s", "frac": achieved / peak,
                         "traffic": traffic, "algorithmic_bytes_per_launch": alg,
                         "launches_per_step": chunks},
            "kernels": dict(phase, scan_shape=shape, wall_ms_per_step=1e3 * t_wall / K),
            "gpu_launches": launches_per_step * K}
    if pipelined:
        # the same kernel over the whole sequence with nothing else running (one-stream step)
        alone_ms = phase["alone"]["scan_ms"]
        alone = scan_bytes_per_head_token(cfg) * units_rank / (alone_ms / 1e3) / 1e9
        line["roofline"]["alone"] = {"achieved": alone, "frac": alone / peak, "ms_per_launch": alone_ms,
                                     "note": "scan kernel over all T tokens, timed alone"}
    line["clocks"] = clk.summary()
    if pipelined:
        line["select_roofline"] = select_roofline(cfg, units_rank, phase["alone"]["select_ms"], line["clocks"])

    if not args.no_e2e:
        line["e2e"] = e2e(st, cfg, sdm, args, dev, torch, K, world)
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        import oracle
        oracle.build()
        line["cpu_baseline"] = cpu_baseline(cfg, wl, oracle)[0]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def huge_page_share(tensors):
    """Share of the host tensors' resident bytes that sit on transparent huge pages (from
    /proc/self/smaps; None where that cannot be read)."""
    import re
    spans = [(t.data_ptr(), t.data_ptr() + t.numel() * t.element_size()) for t in tensors]
    huge = rss = 0
    cur = False
    try:
        with open("/proc/self/smaps") as f:
            for line in f:
                m = re.match(r"([0-9a-f]+)-([0-9a-f]+) ", line)
                if m:
                    lo, hi = int(m.group(1), 16), int(m.group(2), 16)
                    cur = any(a < hi and b > lo for a, b in spans)
                elif cur and line.startswith("AnonHugePages:"):
                    huge += int(line.split()[1]) * 1024
                elif cur and line.startswith("Rss:"):
                    rss += int(line.split()[1]) * 1024
    except OSError:
        return None
    return round(huge / rss, 3) if rss else None


def e2e(st, cfg, sdm, args, dev, torch, K, world):
    """Same metric through the public API with the inputs in pinned host memory: every
    step copies its k', q', v, alpha, beta host->device and its o device->host inside the
    timed region.  Streamed like a serving loop: device inputs and outputs are double
    buffered, so step k+1's host->device copies (on a copy stream) overlap step k's
    compute, and step k's device->host copy overlaps step k+1.  With the pipelined pass a
    step's inputs are copied token window by token window (one window per chunk) and each
    chunk's selection waits only for its own window (sdm_forward_streamed), so the first
    step starts on its first window instead of the whole batch."""
    names = ("kp", "qp", "v", "alpha", "beta")
    # page-locked host buffers on huge pages (sdm.pinned_empty), as a serving loop would keep them
    host = {k: sdm.pinned_empty(st[k].shape, st[k].dtype, dev) for k in names}
    for k in names:
        host[k].copy_(st[k])
    bufs = [{k: st[k] for k in names}, {k: torch.empty_like(st[k]) for k in names}]
    outs = [st["o"], torch.empty_like(st["o"])]
    o_host = [sdm.pinned_empty(st["o"].shape, torch.float32, dev) for _ in range(2)]
    h2d = sum(host[k].numel() * host[k].element_size() for k in names)
    d2h = o_host[0].numel() * 4
    copy = torch.cuda.Stream(device=dev)
    main = torch.cuda.current_stream(dev)
    chunks = sdm.forward_chunks(cfg.T, args.chunks)
    torch.cuda.synchronize(dev)
    # This host's copy rates, alone (context for the streamed number: the loop is copy bound
    # when h2d_bytes_per_step / H2D rate exceeds the device step).
    rates = {}
    for label, dst, src in (("h2d_gbs_alone", bufs[1]["kp"], host["kp"]), ("d2h_gbs_alone", o_host[1], outs[0])):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(copy):
            a.record(copy)
            dst.copy_(src, non_blocking=True)
            b.record(copy)
        torch.cuda.synchronize(dev)
        rates[label] = round(src.numel() * src.element_size() / a.elapsed_time(b) / 1e6, 1)

    pipelined = args.pipeline == "on"
    Tc = -(-cfg.T // chunks)

    def run(n):
        ready = [torch.cuda.Event() for _ in range(n + 1)]
        window = [[torch.cuda.Event() for _ in range(chunks)] for _ in range(n + 1)]
        free = [torch.cuda.Event() for _ in range(n)]       # inputs of step k consumed
        done = [torch.cuda.Event() for _ in range(n)]       # o of step k written
        copy.wait_stream(main)

        def h2d_step(k):
            with torch.cuda.stream(copy):
                if k >= 2:
                    copy.wait_event(free[k - 2])
                if pipelined:
                    for c in range(chunks):
                        t0, t1 = c * Tc, min(cfg.T, (c + 1) * Tc)
                        for name in names:
                            sdm.copy_token_window(bufs[k % 2][name], host[name], t0, t1, stream=copy)
                        window[k][c].record(copy)
                else:
                    for name in names:
                        bufs[k % 2][name].copy_(host[name], non_blocking=True)
                ready[k].record(copy)

        h2d_step(0)
        for k in range(n):
            if not pipelined:
                main.wait_event(ready[k])
            if k + 1 < n:
                h2d_step(k + 1)
            # the inputs are free once the (last) scan kernel starts: selection and planning
            # read them, the scan reads only the planning records
            if args.pipeline == "on":
                sev = [torch.cuda.Event() for _ in range(2 * chunks)]
                sev[2 * chunks - 2] = free[k]
                run_forward(st, cfg, sdm, args, inp=bufs[k % 2], o=outs[k % 2], scan_ev=sev,
                            input_ev=window[k])
            else:
                run_step(st, cfg, sdm, args, inp=bufs[k % 2], o=outs[k % 2],
                         ev=[torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event(), free[k],
                             torch.cuda.Event()])
            done[k].record(main)
            with torch.cuda.stream(copy):
                copy.wait_event(done[k])
                o_host[k % 2].copy_(outs[k % 2], non_blocking=True)
        main.wait_stream(copy)

    run(2)
    torch.cuda.synchronize(dev)
    n = max(2, K)  # the pipeline fill (first step's copies) is amortised over K steps
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    a.record(main)
    run(n)
    b.record(main)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(a.elapsed_time(b), dev)
    return {"value": whole_job_rate(cfg.B * cfg.H * cfg.T, n, world, ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "steps": n, "ms_per_step": ms / n, **rates,
            "host_huge_page_share": huge_page_share(list(host.values()) + o_host),
            "pipeline": "double-buffered: step k+1's host->device copies and step k's device->host copy "
                        "overlap step k's compute (copy stream); inputs copied token window by window, "
                        "each chunk's selection waiting for its own window (sdm_forward_streamed)"
                        if pipelined else
                        "double-buffered: step k+1's host->device copies and step k's device->host copy "
                        "overlap step k's compute (copy stream)"}


def run_stream(args):
    """The streamed long-context workload: each rank's sequences are fed in chunks of
    cfg.chunk tokens with the state carried from chunk to chunk (sdm_forward from M_0 for
    the first chunk, from the state in M for the others).  A step is the whole stream
    (cfg.T tokens).  Every chunk's inputs are drawn in HBM by the device generator just
    before the chunk; the generator runs on the same stream but outside the timed
    intervals, which cover each chunk's forward call alone (its time is reported apart)."""
    import torch
    import torch.distributed as dist

    import sparse_state_linear_sdm_gb300 as sdm
    from sparse_state_linear_sdm_gb300 import workloads as wl

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = workload(args)
    C = cfg.chunk
    n_chunks = -(-cfg.T // C)
    dt = torch.bfloat16 if cfg.in_dtype == "bf16" else torch.float32
    bias = wl.half_bias(cfg)
    bias_d = None if bias is None else torch.from_numpy(bias).to(dev)
    sh = (cfg.B, cfg.H, C)
    inp = dict(kp=torch.empty(sh + (2, cfg.S), dtype=dt, device=dev),
               qp=torch.empty(sh + (2, cfg.S), dtype=dt, device=dev),
               v=torch.empty(sh + (cfg.d_v,), dtype=dt, device=dev),
               alpha=torch.empty(sh, dtype=torch.float32, device=dev),
               beta=torch.empty(sh, dtype=torch.float32, device=dev))
    M0 = sdm.gen_M0(cfg.seed, cfg.H, cfg.N, cfg.d_v, float(wl.M0_SCALE), device=dev)
    M = torch.empty((cfg.B, cfg.H, cfg.N, cfg.d_v), dtype=torch.float32, device=dev)
    sel = (torch.empty(sh + (cfg.W,), dtype=torch.int32, device=dev),
           torch.empty(sh + (cfg.W,), dtype=torch.float32, device=dev),
           torch.empty(sh + (cfg.R,), dtype=torch.int32, device=dev),
           torch.empty(sh + (cfg.R,), dtype=torch.float32, device=dev))
    o = torch.empty(sh + (cfg.d_v,), dtype=torch.float32, device=dev)
    ws = sdm.forward_workspace(cfg.B, cfg.H, C, cfg.d_v, cfg.W, cfg.R, dev, args.chunks)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    sub = sdm.forward_chunks(C, args.chunks)
    E = lambda: torch.cuda.Event(enable_timing=True)

    def chunk_len(c):
        return min(C, cfg.T - c * C)

    def step(ev_gen=None, ev_fwd=None, ev_scan=None):
        for c in range(n_chunks):
            Tc = chunk_len(c)
            part = {k: v[:, :, :Tc] for k, v in inp.items()} if Tc < C else inp
            if ev_gen:
                ev_gen[c][0].record()
            sdm.gen_inputs(cfg.seed, cfg.B, cfg.H, Tc, cfg.S, cfg.d_v, dt, cfg.alpha_lo,
                           0 if cfg.beta_kind == "uniform" else 1, half_bias=bias_d,
                           b_off=rank_batch_offset(rank, cfg.B), t_off=c * C, T_total=cfg.T, out=part)
            if ev_fwd:
                ev_gen[c][1].record()
                ev_fwd[c][0].record()
            sdm.forward(part["kp"], part["qp"], part["v"], part["alpha"], part["beta"], M0 if c == 0 else None,
                        cfg.W, cfg.R, M=M, workspace=ws, dev_err=err, out=sel, o=o, chunks=args.chunks,
                        scan_events=ev_scan[c] if ev_scan else None)
            if ev_fwd:
                ev_fwd[c][1].record()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if err.item() != 0:
        raise RuntimeError(f"device error flags {err.item()}")
    K = args.steps
    ev_gen = [[[E(), E()] for _ in range(n_chunks)] for _ in range(K)]
    ev_fwd = [[[E(), E()] for _ in range(n_chunks)] for _ in range(K)]
    ev_scan = [[[E() for _ in range(2 * sub)] for _ in range(n_chunks)] for _ in range(K)]
    for group in (ev_gen, ev_fwd, ev_scan):
        for per_step in group:
            for per_chunk in per_step:
                for x in per_chunk:
                    x.record()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for k in range(K):
            step(ev_gen[k], ev_fwd[k], ev_scan[k])
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
    if world > 1:
        dist.barrier()
    fwd_ms = sum(a.elapsed_time(b) for per_step in ev_fwd for a, b in per_step)
    gen_ms = sum(a.elapsed_time(b) for per_step in ev_gen for a, b in per_step)
    fwd_ms = max_over_ranks(fwd_ms, dev)
    units_rank = cfg.B * cfg.H * cfg.T
    value = whole_job_rate(units_rank, K, world, fwd_ms)
    launches = [e[2 * j].elapsed_time(e[2 * j + 1]) for per_step in ev_scan for e in per_step
                for j in range(sub)]
    scan_launch_ms = sum(launches) / len(launches)
    units_launch = cfg.B * cfg.H * C / sub
    peak, peak_kind = hbm_peak()
    alg = scan_bytes_per_head_token(cfg) * units_launch
    achieved = alg / (scan_launch_ms / 1e3) / 1e9
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": fwd_ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": dict(config_dict(cfg), chunk=C, chunks_per_stream=n_chunks,
                           step=f"the whole stream: {n_chunks} calls of sdm_forward over {C}-token chunks, the "
                                f"state carried between them (M_0 for the first); each chunk's inputs drawn in HBM "
                                f"by the device generator before its call, outside the timed intervals",
                           l2="state table (2 GB per sequence of 4 heads) and each chunk's k'/q' exceed the "
                              "129 MB L2"),
            "roofline": {"kernel": "sdm scan kernel", "bound": "hbm", "achieved": achieved, "peak": peak,
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                         else "fallback", "unit": "GB/s", "frac": achieved / peak, "traffic": None,
                         "algorithmic_bytes_per_launch": alg, "launches_per_step": n_chunks * sub,
                         "note": f"only {cfg.B * cfg.H} independent scans: latency-bound, not bandwidth-bound"},
            "kernels": {"gen_ms_per_step": gen_ms / K, "forward_ms_per_step": fwd_ms / K,
                        "scan_ms_per_launch": scan_launch_ms, "scan_launches_per_chunk": sub,
                        "us_per_token": 1e3 * fwd_ms / K / cfg.T,
                        "scan_shape": sdm.scan_launch_info(cfg.B, cfg.H, cfg.d_v, cfg.W, cfg.R),
                        "wall_ms_per_step": 1e3 * t_wall / K},
            "gpu_launches": K * n_chunks * (1 + 2 + 3 * sub),
            "e2e": None,
            "e2e_note": "not measured for the stream: its inputs (36 GB per stream) are drawn on the device"}
    line["clocks"] = clk.summary()
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        import oracle
        oracle.build()
        line["cpu_baseline"] = cpu_baseline(cfg, wl, oracle, steps=5)[0]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_decode(args):
    """Single-token decode for a batch of sequences with resident state: K tokens, one
    launch of the single decode kernel (selection, planning, scan) per token."""
    import torch

    import sparse_state_linear_sdm_gb300 as sdm
    from sparse_state_linear_sdm_gb300 import workloads as wl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = workload(args)
    K = max(args.steps, 50)
    st = make_state(dataclasses_replace(cfg, T=K + args.warmup), rank, dev, torch, sdm, wl)
    sdm.init_state_from_M0(st["M"], st["M0"])
    step = sdm.DecodeStep(st["M"], cfg.W, cfg.R, in_dtype=st["kp"].dtype).capture()
    names = ("kp", "qp", "v", "alpha", "beta")
    # Each token's inputs as a producer would hand them over: contiguous tensors of their
    # own (staged before timing).  The single kernel reads them where they are.
    per_token = {k: torch.stack([st[k][:, :, t:t + 1] for t in range(args.warmup + K)]) for k in names}
    # the tensor objects too (a producer hands each token's own tensors over; no slicing in
    # the timed loop)
    token_args = [[per_token[k][t] for k in names] for t in range(args.warmup + K)]

    def token(t):
        return step(*token_args[t])

    def token_strided(t):  # slices of the [B, H, T, ...] inputs: copied into the step's buffers
        return step(*[st[k][:, :, t:t + 1] for k in names])

    for t in range(args.warmup):
        token(t)
        token_strided(t)
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for t in range(args.warmup, args.warmup + K):
        token(t)
    b.record()
    torch.cuda.synchronize(dev)
    ms = a.elapsed_time(b) / K
    a1, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a1.record()
    for t in range(args.warmup, args.warmup + K):
        token_strided(t)
    b1.record()
    torch.cuda.synchronize(dev)
    ms_strided = a1.elapsed_time(b1) / K
    # The same kernels with the inputs already in the step's buffers (a producer that
    # writes them in place): graph replays only, state still advancing token by token.
    a2, b2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a2.record()
    for _ in range(K):
        step.run()
    b2.record()
    torch.cuda.synchronize(dev)
    ms_in_place = a2.elapsed_time(b2) / K
    # Device time per token: one graph of G consecutive tokens (inputs already resident, one
    # launch per token), replayed; the host's per-replay cost is then spread over G tokens.
    G = 16
    toks = {k: torch.stack([st[k][:, :, t:t + 1].contiguous() for t in range(G)])
            for k in ("kp", "qp", "v", "alpha", "beta")}
    sel_g = [torch.empty_like(x) for x in step.sel]
    o_g = torch.empty_like(step.o)
    chain = lambda: [sdm.decode_step(toks["kp"][g], toks["qp"][g], toks["v"][g], toks["alpha"][g],
                                     toks["beta"][g], st["M"], cfg.W, cfg.R, out=sel_g, o=o_g,
                                     table=step.table)
                     for g in range(G)] if step.fused else None
    ms_device = None
    if step.fused:
        chain()
        torch.cuda.synchronize(dev)
        gph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gph):
            chain()
        gph.replay()
        torch.cuda.synchronize(dev)
        reps = max(K // G, 4)
        a3, b3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a3.record()
        for _ in range(reps):
            gph.replay()
        b3.record()
        torch.cuda.synchronize(dev)
        ms_device = a3.elapsed_time(b3) / (reps * G)
    state_bytes = cfg.B * cfg.H * (2 * cfg.W + cfg.R) * cfg.d_v * 4
    line = {"metric": "SDM decode head-tokens/s (one token per step, state resident)",
            "value": cfg.B * cfg.H / (ms / 1e3), "unit": "head-tokens/s", "n_gpus": 1, "steps": K,
            "warmup": args.warmup, "us_per_step": ms * 1e3, "higher_is_better": True, "dtype": "f32",
            "data": "synthetic", "config": dict(config_dict(cfg), T=1, step="decode: CUDA graph of select + plan + scan"),
            "state_bytes_per_step": state_bytes, "state_gbs": state_bytes / (ms / 1e3) / 1e9,
            "us_per_step_inputs_in_place": ms_in_place * 1e3,
            "us_per_step_strided_inputs": ms_strided * 1e3,
            "us_per_step_device": ms_device * 1e3 if ms_device is not None else None,
            "decode_kernel": "one fused kernel per token" if step.fused else "select + plan + scan",
            "note": "us_per_step: DecodeStep called per token on that token's own contiguous inputs (tensor "
                    "objects staged before timing) "
                    "(one launch of the single kernel, which reads them where they are); "
                    "us_per_step_strided_inputs: called on slices of the [B, H, T, ...] inputs, which are "
                    "copied into the step's buffers (5 copies) before the captured graph runs; "
                    "us_per_step_inputs_in_place replays the one-token graph alone on inputs already there "
                    "(bounded by the host's graph launches); us_per_step_device replays a graph of 16 "
                    "consecutive tokens (device time per token)",
            "gpu_launches": (1 if step.fused else 3) * K}
    print(json.dumps(line), flush=True)


def backward_bytes_per_head_token(cfg) -> int:
    """Algorithmic bytes of the backward scan per head-token: dO; the stored write rows
    (before their update) and read rows; the adjoint rows gathered and scattered at every
    write and read slot; v, alpha, beta; slots and scores; dv (fp32 d_v-vectors)."""
    K = cfg.W + cfg.R
    elt = 2 if cfg.in_dtype == "bf16" else 4
    return cfg.d_v * 4 + K * cfg.d_v * 4 + 2 * K * cfg.d_v * 4 + cfg.d_v * elt + 8 + K * 8 + cfg.d_v * 4


def zero_adjoint_slots(sel, N, torch):
    """Under a zero final adjoint: the write slots and read slots whose adjoint row is still
    zero (no later read selects the row; a read at the same token comes after the token's
    writes).  Counted with torch on the device from the slots alone (measurement only)."""
    iw, ir = sel[0], sel[2]
    B, H, T, W = iw.shape
    R = ir.shape[3]
    dev = iw.device
    tr = torch.arange(T, device=dev).repeat_interleave(R)
    t = torch.arange(T, device=dev)[:, None]
    zw = zr = 0
    for b in range(B):
        for h in range(H):
            last = torch.full((N,), -1, dtype=torch.int64, device=dev)
            last.scatter_reduce_(0, ir[b, h].reshape(-1).long(), tr, reduce="amax")
            zr += int((last[ir[b, h].long()] == t).sum())
            zw += int((last[iw[b, h].long()] < t).sum())
    return zw, zr


def run_backward(args):
    """Training backward of one forward pass: with the forward's stored rows, K steps of
    (reverse scan with a zero final adjoint -- the loss reads the outputs only -- with the
    finish and the batch reduction into dM_0; half gradients of k' and q').  The same
    steps with the adjoint table cleared and the full reverse scan are timed beside it."""
    import torch

    import sparse_state_linear_sdm_gb300 as sdm
    from sparse_state_linear_sdm_gb300 import workloads as wl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = workload(args)
    st = make_state(cfg, rank, dev, torch, sdm, wl)
    del st["fws"]
    sel = st["sel"]
    sdm.select(st["kp"], st["qp"], cfg.W, cfg.R, out=sel)
    sdm.init_state_from_M0(st["M"], st["M0"])
    E = lambda: torch.cuda.Event(enable_timing=True)
    f0, f1 = E(), E()
    f0.record()
    o, w_prev, r_rows = sdm.scan_forward_train(st["M"], *sel, st["v"], st["alpha"], st["beta"], o=st["o"],
                                               workspace=st["ws"], dev_err=st["err"])
    f1.record()
    gen = torch.Generator(device=dev).manual_seed(cfg.seed)
    dO = torch.randn((cfg.B, cfg.H, cfg.T, cfg.d_v), generator=gen, device=dev)
    G = st["M"]   # the state is not needed any more: its buffer holds the adjoint
    ws = torch.empty(sdm.backward_workspace_size(cfg.B, cfg.H, cfg.T, cfg.N, cfg.d_v, cfg.W, cfg.R, True),
                     dtype=torch.uint8, device=dev)
    dkp = torch.empty((cfg.B, cfg.H, cfg.T, 2, cfg.S), device=dev)
    dqp = torch.empty_like(dkp)

    def step(final_zero, ev=None):
        if ev:
            ev[0].record()
        if not final_zero:
            sdm.fill_state(G, 0.0)
        if ev:
            ev[1].record()
        g = sdm.scan_backward(*sel, st["v"], st["alpha"], st["beta"], w_prev, r_rows, dO, G, workspace=ws,
                              final_zero=final_zero, dm0_only=final_zero)
        if ev:
            ev[2].record()
        sdm.select_backward(sel[0], g["dsc_w"], cfg.S, out=dkp)
        sdm.select_backward(sel[2], g["dsc_r"], cfg.S, out=dqp)
        if ev:
            ev[3].record()

    def timed(final_zero):
        for _ in range(args.warmup):
            step(final_zero)
        torch.cuda.synchronize(dev)
        evs = [[E() for _ in range(4)] for _ in range(args.steps)]
        with ClockSampler(local) as clk:
            for k in range(args.steps):
                step(final_zero, evs[k])
            torch.cuda.synchronize(dev)
        K = args.steps
        return dict(total=evs[0][0].elapsed_time(evs[-1][3]),
                    zero_ms=sum(e[0].elapsed_time(e[1]) for e in evs) / K,
                    scan_ms=sum(e[1].elapsed_time(e[2]) for e in evs) / K,
                    sel_ms=sum(e[2].elapsed_time(e[3]) for e in evs) / K), clk

    lazy, clk = timed(True)
    full, _ = timed(False)
    K = args.steps
    units = cfg.B * cfg.H * cfg.T
    peak, peak_kind = hbm_peak()
    row = cfg.d_v * 4
    zw, zr = zero_adjoint_slots(sel, cfg.N, torch)
    # A zero read slot skips its adjoint load; a zero write slot its adjoint load and store
    # and its stored row's load; every token reads its words of zero bits.
    alg_full = backward_bytes_per_head_token(cfg) * units
    alg = alg_full - zr * row - 3 * zw * row + units * 4 * ((cfg.W + cfg.R + 31) // 32)
    achieved = alg / (lazy["scan_ms"] / 1e3) / 1e9
    achieved_full = alg_full / (full["scan_ms"] / 1e3) / 1e9
    slots_w, slots_r = units * cfg.W, units * cfg.R
    line = {"metric": "SDM backward head-tokens/s on 1 GB300 (reverse scan, score and half gradients)",
            "value": whole_job_rate(units, K, world, lazy["total"]), "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": lazy["total"] / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(config_dict(cfg), step="backward with a zero final adjoint (dL/dM_T = 0): reverse "
                                                  "scan + finish + dM0 reduction (sdm_scan_backward_ex, "
                                                  "SDM_BWD_FINAL_ZERO), select backward for k' and q'"),
            "roofline": {"kernel": "sdm_scan_backward_ex (zero-slot passes, reverse scan, finish, batch reduction)",
                         "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "algorithmic_bytes_per_launch": alg, "traffic": None,
                         "note": "bytes of the reverse scan with the zero slots' rows left out, over the whole "
                                 "call's time",
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured"
                         else "fallback"},
            "kernels": {"forward_train_ms": f0.elapsed_time(f1), "scan_backward_ms": lazy["scan_ms"],
                        "select_backward_ms": lazy["sel_ms"],
                        "zero_slots": {"write": zw / slots_w, "read": zr / slots_r},
                        "cleared_adjoint": {"ms_per_step": full["total"] / K, "fill_ms": full["zero_ms"],
                                            "scan_backward_ms": full["scan_ms"], "select_backward_ms": full["sel_ms"],
                                            "algorithmic_bytes_per_launch": alg_full,
                                            "achieved_gbs": achieved_full, "frac": achieved_full / peak}},
            "gpu_launches": 8 * K, "clocks": clk.summary()}
    if rank == 0:
        print(json.dumps(line), flush=True)


def bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def run_project(args):
    """The projections x -> k', q' of every token of the workload: one tensor-core GEMM
    [B*T, D] x [D, 4*H*S] per step, bf16 outputs in the selection's layout."""
    import numpy as np
    import torch

    import sparse_state_linear_sdm_gb300 as sdm
    from sparse_state_linear_sdm_gb300 import workloads as wl

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = workload(args)
    D = args.dmodel or wl.PROJ_D
    B, T, H, S = cfg.B, cfg.T, cfg.H, cfg.S
    b0 = rank_batch_offset(rank, B)
    xb = wl.projection_features(cfg.seed, B * world, T, D, b0 * T, (b0 + B) * T)
    wb = wl.projection_weights(cfg.seed, H, S, D)
    to_dev = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)
    x = to_dev(xb).view(B, T, D)
    w = to_dev(wb)
    kp = torch.empty((B, H, T, 2, S), dtype=torch.bfloat16, device=dev)
    qp = torch.empty_like(kp)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    for _ in range(args.warmup):
        sdm.project_kq(x, w, H, S, out=(kp, qp), dev_err=err, max_ctas=args.max_ctas, pair=args.pair)
    torch.cuda.synchronize(dev)
    K = args.steps
    E = lambda: torch.cuda.Event(enable_timing=True)
    evs = [(E(), E()) for _ in range(K)]
    with ClockSampler(local) as clk:
        for a, b in evs:
            a.record()
            sdm.project_kq(x, w, H, S, out=(kp, qp), dev_err=err, max_ctas=args.max_ctas, pair=args.pair)
            b.record()
        torch.cuda.synchronize(dev)
    if err.item() != 0:
        raise RuntimeError(f"projection kernel reported device error bits {err.item()}")
    total = evs[0][0].elapsed_time(evs[-1][1])
    per = [a.elapsed_time(b) for a, b in evs]
    ms = statistics.mean(per)
    max_ms = max_over_ranks(total, dev)
    flops = 2.0 * B * T * D * 4 * H * S
    achieved = flops / (ms / 1e3) / 1e12
    peak, peak_kind = bf16_peak()
    line = {"metric": "SDM k'/q' projection head-tokens/s on 1 GB300 (tensor-core GEMM)",
            "value": whole_job_rate(B * H * T, K, world, max_ms), "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": total / K, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 (fp32 accumulation)", "data": "synthetic",
            "config": {"workload": f"{cfg.name}: x [B={B}, T={T}, D={D}] bf16 -> k', q' [B, H={H}, T, 2, S={S}] bf16",
                       "gemm": [B * T, 4 * H * S, D], "l2": "inputs larger than L2 (x is "
                       f"{B * T * D * 2 / 1e6:.0f} MB, outputs {2 * B * H * T * 2 * S * 2 / 1e9:.1f} GB)"},
            "roofline": {"kernel": "sdm project_kernel (tcgen05.mma kind::f16, TMA, TMEM)", "bound": "tensor",
                         "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                         "algorithmic_flops_per_launch": flops,
                         "traffic": project_traffic([B * T, 4 * H * S, D], args),
                         "algorithmic_bytes_per_launch": 2.0 * (B * T * D + 4 * H * S * D + B * T * 4 * H * S),
                         "peak_source": f"{peak_kind} (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst)"
                         if peak_kind == "measured" else "fallback 1.9 PFLOP/s"},
            "kernel_ms": {"mean": ms, "min": min(per), "max": max(per)},
            "launch": {"max_ctas": args.max_ctas, "pair": args.pair},
            "gpu_launches": K, "clocks": clk.summary()}
    line["fused"] = project_select_timing(sdm, torch, x, w, kp, qp, cfg, H, S, K, args.warmup, dev, ms, peak)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        n = 32
        xs = wl.bf16_to_f32(xb[:n])
        ws = wl.bf16_to_f32(wb)
        t0 = time.perf_counter()
        reps = 0
        while reps < 3 or time.perf_counter() - t0 < 2.0:
            oracle.project(xs, ws, H, S)
            reps += 1
        dt = (time.perf_counter() - t0) / reps
        line["cpu_baseline"] = {"value": n * H / dt, "unit": UNIT, "cores": os.cpu_count() or 1,
                                "kind": "oracle", "sample": f"oracle.project (fp64 matmul) on {n} tokens x "
                                f"{4 * H * S} columns x D={D}, mean of {reps}"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def project_select_timing(sdm, torch, x, w, kp, qp, cfg, H, S, K, warmup, dev, project_ms, peak):
    """The projections fused with the selection (sdm_project_select: k', q' never in device
    memory) against the unfused pair (sdm_project_kq, then sdm_select on its output), each
    timed over K launches after `warmup`; the two must give the same slots and scores."""
    W, R = cfg.W, cfg.R
    B, T = x.shape[0], x.shape[1]
    E = lambda: torch.cuda.Event(enable_timing=True)
    sel = sdm.select(kp, qp, W, R)
    ws = sdm.project_select_workspace(B, T, H, S, W, R, dev)
    fused = sdm.project_select(x, w, H, S, W, R, workspace=ws)
    torch.cuda.synchronize(dev)
    same = all(torch.equal(a, b) for a, b in zip(fused, sel))

    def timed(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize(dev)
        evs = [(E(), E()) for _ in range(K)]
        for a, b in evs:
            a.record()
            fn()
            b.record()
        torch.cuda.synchronize(dev)
        return statistics.mean(a.elapsed_time(b) for a, b in evs)

    sel_ms = timed(lambda: sdm.select(kp, qp, W, R, out=sel))
    fused_ms = timed(lambda: sdm.project_select(x, w, H, S, W, R, out=fused, workspace=ws))
    kq_bytes = 2 * kp.numel() * kp.element_size()
    lists_bytes = sdm.lib().sdm_project_select_workspace_size(B, T, H, S, W, R)
    flops = 2.0 * B * T * x.shape[2] * 4 * H * S
    return {"project_select_ms": fused_ms, "project_ms": project_ms, "select_ms": sel_ms,
            "unfused_ms": project_ms + sel_ms, "bit_identical_to_unfused": same,
            "fused_tflops": flops / (fused_ms / 1e3) / 1e12, "peak_tflops": peak,
            "kq_bytes_not_written": kq_bytes, "inner_list_bytes": lists_bytes,
            "note": "fused: one kernel projects on the tensor cores and takes each half's top-k on "
                    "chip (per-half lists, 4 B per entry, written instead of k' and q'), then the "
                    "outer top-K kernel; unfused: sdm_project_kq writes k', q' (bf16) and sdm_select "
                    "reads them back"}


def dataclasses_replace(cfg, **kw):
    import dataclasses

    return dataclasses.replace(cfg, **kw)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    elif args.mode == "decode":
        run_decode(args)
    elif args.mode == "backward":
        run_backward(args)
    elif args.mode == "project":
        run_project(args)
    elif workload(args).chunk:
        run_stream(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
