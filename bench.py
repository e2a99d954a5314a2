"""Benchmark: selective scan (S6) forward on one B300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one ss_scan_fwd over the Mamba-2.8B block shape (batch 8, d_inner
5120, d_state 16, L 2048; bf16 u/delta/z/B/C, fp32 state and output, z gate
and D skip on, final state written). Inputs are seeded synthetic draws
(workloads.CONFIGS["mamba2p8b"]); 843 MB move per step, more than the 126 MB
L2, so no flush is needed between steps.

Prints one JSON line. `value` is elements/s (batch * d_inner * L per second)
with inputs resident in HBM, summed over ranks; `e2e` repeats the metric with
host buffers (pinned H2D of the inputs and D2H of y and h_last inside the
timed region); `roofline` compares the kernel with the HBM and ALU floors;
`cpu_baseline` times the fp64 oracle on a bounded sample on the host cores.
Under torchrun every rank runs its own replica (rows are independent: no
collective on the data path); only the timing is reduced (max over ranks).

--impl reference times the fp64 CPU oracle itself (the only reference this
project has) on the same metric, as a bounded row sample per step.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

CONFIG = "mamba2p8b"
MAX_SM_MHZ = 2032.0        # B300 maximum SM clock
FALLBACK_HBM_GBS = 6400.0  # used only when MEASURED_PEAKS.json is absent
FP32_LANES_PER_SM = 128    # FMA-pipe lanes per SM per clock
METRIC = "selective-scan elements/s (B*D*L) and HBM GB/s as % of roofline"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=CONFIG)
    ap.add_argument("--variant", default="auto", choices=["auto", "rows", "chunked", "simple"])
    ap.add_argument("--tpr", type=int, default=0, help="threads per row (rows variant)")
    ap.add_argument("--segments", type=int, default=0)
    ap.add_argument("--skip-cpu", action="store_true", help="skip the oracle CPU baseline")
    ap.add_argument("--skip-e2e", action="store_true", help="skip the host-buffer e2e leg")
    ap.add_argument("--skip-probe", action="store_true", help="skip the ALU-rate probes")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--skip-decode", action="store_true", help="skip the decode-step leg")
    ap.add_argument("--skip-conv", action="store_true", help="skip the conv1d leg")
    ap.add_argument("--skip-bwd", action="store_true", help="skip the backward leg")
    ap.add_argument("--skip-ssd", action="store_true", help="skip the Mamba-2 SSD leg")
    ap.add_argument("--skip-configs", action="store_true",
                    help="skip the mamba130m and long1m scan legs")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(pg, value, device):
    """The largest of every rank's `value` (a job's timed region lasts as long
    as its slowest rank's); `value` itself when there is one rank (pg None).
    `pg` is torch.distributed with any backend; `device` is where that
    backend's tensors live (a GPU for NCCL, the CPU for gloo)."""
    if pg is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world, units_per_rank, steps, max_ms):
    """Whole-job units per second: every rank processed `units_per_rank` per
    step (replicas, weak scaling) within the slowest rank's `max_ms`."""
    return world * units_per_rank * steps / (max_ms * 1e-3)


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def step_bytes(cfg, out_bytes=4):
    """Algorithmic bytes of one scan: read u, delta, z, B, C once; write y and
    h_last; read A, D, delta_bias."""
    esz = 2 if cfg.in_dtype == "bf16" else 4
    bdl = cfg.batch * cfg.dim * cfg.seqlen
    bnl = cfg.batch * cfg.dstate * cfg.seqlen
    return (3 * bdl * esz + 2 * bnl * esz + bdl * out_bytes
            + cfg.batch * cfg.dim * cfg.dstate * 4 + cfg.dim * cfg.dstate * 4 + 2 * cfg.dim * 4)


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return float(d["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------- CPU oracle timing

_ORACLE_BLOCKS = {}


def time_oracle(cfg, seconds, threads, max_blocks=2):
    """Time the fp64 oracle on cfg's rows for about `seconds` of host time.

    The sample is the first `max_blocks` blocks of up to 4096 rows (every row
    at full length L); they are scanned in turn, repeatedly, until the timed
    total passes `seconds`. Inputs are generated once per block, outside the
    timed region. Returns (elements/s, row scans timed, distinct rows, elapsed)."""
    import oracle
    oracle.build()
    block = max(1, min(cfg.rows, 4096))
    starts = list(range(0, min(cfg.rows, block * max_blocks), block))
    timed, done, i = 0.0, 0, 0
    while True:
        key = (cfg.name, starts[i % len(starts)])
        if key not in _ORACLE_BLOCKS:
            rows = np.arange(key[1], min(key[1] + block, cfg.rows))
            _ORACLE_BLOCKS[key] = (rows, workloads.scan_inputs(cfg, rows=rows))
        rows, inp = _ORACLE_BLOCKS[key]
        t0 = time.perf_counter()
        oracle.scan_fwd(inp["u"], inp["delta"], inp["A"], inp["B"], inp["C"], D=inp["D"],
                        delta_bias=inp["delta_bias"], z=inp["z"], rows=rows, dim=cfg.dim,
                        threads=threads)
        timed += time.perf_counter() - t0
        done += len(rows)
        i += 1
        if timed >= seconds:
            break
    distinct = min(cfg.rows, block * len(starts))
    return done * cfg.seqlen / timed, done, distinct, timed


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self, t0, t1):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons, n = [], None, set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            if not (t0 - 0.15 <= ts <= t1 + 0.15):
                continue
            n += 1
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() in ("active", "1"):
                    reasons.add(nm)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": n}


# ---------------------------------------------------------------- ALU probe

def probe_alu(device):
    import ctypes
    path = os.path.join(ROOT, "selective_state_space_136_b300", "libss_probe.so")
    lib = ctypes.CDLL(path)
    lib.ss_probe_alu.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                 ctypes.POINTER(ctypes.c_double)]
    out = {}
    for which, name in ((0, "ex2"), (1, "ffma"), (2, "ffma2"), (3, "mixed"), (4, "mma_sync_bf16")):
        r, g = ctypes.c_double(), ctypes.c_double()
        rc = lib.ss_probe_alu(which, device, ctypes.byref(r), ctypes.byref(g))
        out[name] = {"ops_per_s": r.value, "sm_ghz": g.value, "rc": rc}
    # the scan's inner step without memory traffic, at the parallelism shapes
    # allow: 2 rows per lane pair with 8 warps per SM (32-row warps: the 2.8B
    # shape's 40960 rows fill 1184 warps once), 4 rows per lane pair with 4 or
    # 8 warps per SM (64-row warps)
    lib.ss_probe_scan_step.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.POINTER(ctypes.c_double),
                                       ctypes.POINTER(ctypes.c_double)]
    steps = {}
    for rows, warps in ((2, 8), (2, 16), (4, 4), (4, 8)):
        r, g = ctypes.c_double(), ctypes.c_double()
        rc = lib.ss_probe_scan_step(rows, warps, device, ctypes.byref(r), ctypes.byref(g))
        steps["rows%d_warps%d" % (rows, warps)] = {
            "elements_per_clk_per_sm": r.value, "frac_of_ex2_peak": r.value / 32.0,
            "sm_ghz": g.value, "rc": rc}
    out["scan_step"] = steps
    return out


# ---------------------------------------------------------------- traffic from committed ncu summary

def kernel_source_sha():
    h = hashlib.sha256()
    for f in ("ss_pair.cu", "ss_common.cuh"):
        h.update(open(os.path.join(ROOT, "selective_state_space_136_b300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(cfg_name):
    """dram bytes per launch recorded in profiles/, if taken on this exact source."""
    p = os.path.join(ROOT, "profiles", "ncu_scan_pair_%s.md" % cfg_name)
    if not os.path.exists(p):
        return None
    sha, traffic = None, None
    for line in open(p):
        if line.startswith("source_sha:"):
            sha = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_launch:"):
            try:
                traffic = float(line.split(":", 1)[1].strip())
            except ValueError:
                traffic = None
    return traffic if sha == kernel_source_sha() else None


# ---------------------------------------------------------------- our arm

def workload_config(cfg):
    """The `config` keys both arms share: the workload and its sizes."""
    return {"workload": "%s: batch %d, d_inner %d, d_state %d, L %d, %s u/delta/z/B/C, "
                        "fp32 state/y, z gate + D skip, h_last out"
                        % (cfg.name, cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen, cfg.in_dtype),
            "batch": cfg.batch, "d_inner": cfg.dim, "d_state": cfg.dstate,
            "seq_len": cfg.seqlen, "in_dtype": cfg.in_dtype, "out_dtype": "f32"}


def time_decode(ss, ctx, dev, stream, args, n_sets=6):
    """Time ss_state_update on the decode workload (batch 128, d_inner 5120,
    d_state 16, bf16 x/dt/z/B/C, fp32 state in place, fp32 y).

    The 41.9 MB state fits in L2, so `n_sets` independent (state, inputs) sets
    are cycled: between two uses of one state, the other sets move more than
    the 126 MB of L2 through it, and every step reads its state from HBM."""
    import torch
    cfg = workloads.DECODE
    prm = workloads.params(cfg)
    A = torch.from_numpy(prm["A"]).to(dev)
    Dp = torch.from_numpy(prm["D"]).to(dev)
    bias = torch.from_numpy(prm["delta_bias"]).to(dev)

    def bf(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)

    sets = []
    for k in range(n_sets):
        st = torch.from_numpy(workloads.decode_state0(cfg)).to(dev)
        inp = {n: bf(v).to(dev) for n, v in workloads.decode_step_inputs(cfg, k).items()}
        y = torch.empty((cfg.batch, cfg.dim), dtype=torch.float32, device=dev)
        sets.append((st, inp, y))

    # each step's arguments marshalled once (a decode step is shorter than the
    # Python checks of the per-call binding)
    import ctypes
    fn = ss.lib().ss_state_update
    sp = ctypes.c_void_p(stream.cuda_stream)
    prepared = []
    for st, inp, y in sets:
        a = ss.UpdateArgs(cfg.batch, cfg.dim, cfg.dstate, 1, 0, st.data_ptr(), inp["x"].data_ptr(),
                          inp["dt"].data_ptr(), inp["z"].data_ptr(), A.data_ptr(),
                          inp["B"].data_ptr(), inp["C"].data_ptr(), Dp.data_ptr(),
                          bias.data_ptr(), 1, y.data_ptr())
        prepared.append((a, ctypes.byref(a)))

    def one(k):
        if fn(ctx.handle, prepared[k % n_sets][1], sp) != 0:
            raise RuntimeError("ss_state_update failed")

    for k in range(max(args.warmup, 3) * n_sets):
        one(k)
    torch.cuda.synchronize(dev)
    steps = max(args.steps, 1) * n_sets
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for k in range(steps):
        one(k)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if ctx.device_error() != ss.SS_OK:
        raise RuntimeError("device error in the decode leg")
    us = e0.elapsed_time(e1) * 1e3 / steps
    rows = cfg.batch * cfg.dim
    nbytes = (2 * rows * cfg.dstate * 4 + 3 * rows * 2 + 2 * cfg.batch * cfg.dstate * 2
              + rows * 4 + cfg.dim * cfg.dstate * 4 + 2 * cfg.dim * 4)
    gbs = nbytes / (us * 1e-6) / 1e9
    peak, src = measured_peaks()
    return {"workload": "decode: batch %d, d_inner %d, d_state %d, bf16 x/dt/z/B/C, fp32 state "
                        "in place, fp32 y; %d state sets cycled" % (cfg.batch, cfg.dim, cfg.dstate,
                                                                    n_sets),
            "us_per_step": us, "tokens_per_s": cfg.batch / (us * 1e-6),
            "algorithmic_bytes_per_step": nbytes, "gbs": gbs,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "peak_source": src,
                         "unit": "GB/s", "frac": gbs / peak},
            "steps": steps, "gpu_launches": steps}


def time_conv1d(ss, ctx, dev, stream, cfg, args):
    """Time ss_conv1d_fwd, the Mamba block's causal depthwise convolution
    (width 4, silu), over the scan workload's (batch, d_inner, L) in its input
    dtype, output in the same dtype, zero initial state, final state out."""
    import ctypes
    import torch
    W = 4
    g = torch.Generator(device="cpu").manual_seed(cfg.seed)
    dt = torch.bfloat16 if cfg.in_dtype == "bf16" else torch.float32
    x = torch.randn((cfg.batch, cfg.dim, cfg.seqlen), generator=g).to(dt).to(dev)
    w = torch.randn((cfg.dim, W), generator=g).to(dev)
    b = torch.randn((cfg.dim,), generator=g).to(dev)
    out = torch.empty_like(x)
    fs = torch.empty((cfg.batch, cfg.dim, W - 1), device=dev)
    a = ss.Conv1dArgs(cfg.batch, cfg.dim, W, cfg.seqlen, 1 if dt == torch.bfloat16 else 0,
                      1 if dt == torch.bfloat16 else 0, x.data_ptr(), w.data_ptr(),
                      b.data_ptr(), None, 1, out.data_ptr(), fs.data_ptr())
    fn, argp = ss.lib().ss_conv1d_fwd, ctypes.byref(a)
    sp = ctypes.c_void_p(stream.cuda_stream)
    for _ in range(max(args.warmup, 3)):
        assert fn(ctx.handle, argp, sp) == 0
    torch.cuda.synchronize(dev)
    steps = max(args.steps, 1)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn(ctx.handle, argp, sp)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    us = e0.elapsed_time(e1) * 1e3 / steps
    esz = 2 if dt == torch.bfloat16 else 4
    nbytes = cfg.elements * 2 * esz + cfg.rows * (W - 1) * 4 + cfg.dim * (W + 1) * 4
    gbs = nbytes / (us * 1e-6) / 1e9
    peak, src = measured_peaks()
    return {"workload": "conv1d: batch %d, d_inner %d, L %d, width %d, %s in/out, silu, "
                        "final state out" % (cfg.batch, cfg.dim, cfg.seqlen, W, cfg.in_dtype),
            "us_per_call": us, "elements_per_s": cfg.elements / (us * 1e-6),
            "algorithmic_bytes": nbytes, "gbs": gbs,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "peak_source": src,
                         "unit": "GB/s", "frac": gbs / peak},
            "steps": steps, "gpu_launches": steps}


def time_conv_scan(ss, ctx, dev, stream, cfg, d, params, args, probes):
    """The width-4 causal convolution fused in front of the scan (x in, y out)
    against the same two steps as separate calls (conv1d writing u in the input
    dtype, then the scan reading it), on the benchmark workload's tensors."""
    import torch
    g = torch.Generator(device="cpu").manual_seed(12)
    W = 4
    w = (torch.randn(cfg.dim, W, generator=g) * 0.5).to(dev)
    b = (torch.randn(cfg.dim, generator=g) * 0.1).to(dev)
    shp = (cfg.batch, cfg.dim, cfg.seqlen)
    y = torch.empty(shp, dtype=torch.float32, device=dev)
    hl = torch.empty((cfg.batch, cfg.dim, cfg.dstate), dtype=torch.float32, device=dev)
    cs = torch.empty((cfg.batch, cfg.dim, W - 1), dtype=torch.float32, device=dev)
    fused = ss.PreparedConvScan(d["u"], w, d["delta"], params["A"], d["B"], d["C"], ctx=ctx,
                                stream=stream, conv_bias=b, D=params["D"],
                                delta_bias=params["delta_bias"], z=d["z"], y=y, h_last=hl,
                                conv_state_out=cs)
    u = torch.empty_like(d["u"])
    scan = ss.PreparedScan(u, d["delta"], params["A"], d["B"], d["C"], D=params["D"],
                           delta_bias=params["delta_bias"], z=d["z"], y=y, h_last=hl, ctx=ctx,
                           stream=stream)

    def separate():
        ss.ss_conv1d_fwd(d["u"], w, bias=b, silu=True, out=u, final_state=cs, ctx=ctx,
                         stream=stream)
        scan()

    def timed(fn, n):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / n * 1e-3

    n = max(5, min(args.steps, 20))
    t_f = timed(fused, n)
    variant, launches = ctx.last_launch()
    t_s = timed(separate, n)
    if ctx.device_error() != ss.SS_OK:
        raise RuntimeError("device error in the conv+scan leg")
    esz = 2 if cfg.in_dtype == "bf16" else 4
    scan_bytes = step_bytes(cfg)
    conv_state_bytes = cfg.batch * cfg.dim * (W - 1) * 4
    fused_bytes = scan_bytes + conv_state_bytes + cfg.dim * (W + 1) * 4
    u_round_trip = 2 * cfg.elements * esz
    rf = scan_roofline(cfg, t_f, probes, sms_of(dev))
    return {"workload": "conv1d (width 4, bias, silu) fused in front of the scan: " +
                        workload_config(cfg)["workload"],
            "us_fused": t_f * 1e6, "us_separate": t_s * 1e6,
            "elements_per_s_fused": cfg.elements / t_f,
            "algorithmic_bytes_fused": fused_bytes,
            "algorithmic_bytes_separate": fused_bytes + u_round_trip,
            "bytes_saved": u_round_trip,
            "roofline_scan_terms": {"bound": rf["bound"], "term": rf["term"],
                                    "frac_of_floor": rf["frac_of_floor"],
                                    "floor_us": rf["floor_us"],
                                    "note": "the scan's own floor (the convolution adds 4 FMAs "
                                            "and a silu per (b, d, l))"},
            "launches_fused": launches, "steps": n, "gpu_launches": n * (launches + 3)}


def time_bwd(ss, ctx, dev, stream, cfg, d, params, args):
    """Time ss_scan_bwd on the scan workload (the forward inputs already on the
    device, dy fp32, all gradients requested)."""
    import ctypes
    import torch
    L, N = cfg.seqlen, cfg.dstate
    dy = torch.randn((cfg.batch, cfg.dim, L), device=dev)
    f32 = dict(dtype=torch.float32, device=dev)
    g = [torch.empty((cfg.batch, cfg.dim, L), **f32) for _ in range(3)]
    gA = torch.empty((cfg.dim, N), **f32)
    gB, gC = (torch.empty((cfg.batch, N, L), **f32) for _ in range(2))
    gD, gb = (torch.empty((cfg.dim,), **f32) for _ in range(2))
    a = ss.ScanBwdArgs(cfg.batch, cfg.dim, N, L, 1 if cfg.in_dtype == "bf16" else 0,
                       d["u"].data_ptr(), d["delta"].data_ptr(), d["z"].data_ptr(),
                       params["A"].data_ptr(), d["B"].data_ptr(), d["C"].data_ptr(),
                       params["D"].data_ptr(), params["delta_bias"].data_ptr(), 1, None,
                       dy.data_ptr(), None, g[0].data_ptr(), g[1].data_ptr(), g[2].data_ptr(),
                       gA.data_ptr(), gB.data_ptr(), gC.data_ptr(), gD.data_ptr(), gb.data_ptr(),
                       None)
    fn, argp = ss.lib().ss_scan_bwd, ctypes.byref(a)
    sp = ctypes.c_void_p(stream.cuda_stream)
    for _ in range(2):
        assert fn(ctx.handle, argp, sp) == 0
    torch.cuda.synchronize(dev)
    steps = max(1, min(args.steps, 5))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn(ctx.handle, argp, sp)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if ctx.device_error() != ss.SS_OK:
        raise RuntimeError("device error in the backward leg")
    us = e0.elapsed_time(e1) * 1e3 / steps
    esz = 2 if cfg.in_dtype == "bf16" else 4
    # read u, delta, z, dy and B, C; write du, ddelta, dz, dB, dC (fp32)
    nbytes = cfg.elements * (3 * esz + 4 + 3 * 4) + cfg.batch * N * L * (2 * esz + 2 * 4)
    gbs = nbytes / (us * 1e-6) / 1e9
    peak, src = measured_peaks()
    return {"workload": "scan backward: batch %d, d_inner %d, d_state %d, L %d, %s inputs, fp32 "
                        "dy and gradients, all gradients" % (cfg.batch, cfg.dim, N, L,
                                                            cfg.in_dtype),
            "us_per_call": us, "elements_per_s": cfg.elements / (us * 1e-6),
            "algorithmic_bytes": nbytes, "gbs": gbs, "hbm_frac": gbs / peak,
            "hbm_peak_source": src, "steps": steps, "gpu_launches": steps}


def time_ssd(ss, ctx, dev, stream, args, batch=8, L=2048, H=80, P=64, N=128, probes=None):
    """Time ss_ssd_fwd on the Mamba-2 block shape (d_inner 5120 = 80 heads of
    64, d_state 128), bf16 inputs, fp32 y."""
    import ctypes
    import torch
    g = torch.Generator(device="cpu").manual_seed(7)
    bf = torch.bfloat16
    x = torch.randn((batch, L, H, P), generator=g).to(bf).to(dev)
    dt = (torch.randn((batch, L, H), generator=g) * 0.5 - 1.0).to(bf).to(dev)
    Bm = (torch.randn((batch, L, N), generator=g) * 0.3).to(bf).to(dev)
    Cm = (torch.randn((batch, L, N), generator=g) * 0.3).to(bf).to(dev)
    A = -(torch.rand((H,), generator=g) * 3.5 + 0.5).to(dev)
    D = torch.randn((H,), generator=g).to(dev)
    bias = torch.full((H,), -4.0).to(dev)
    y = torch.empty((batch, L, H, P), device=dev)
    hl = torch.empty((batch, H, P, N), device=dev)
    a = ss.SsdArgs(batch, H, P, N, L, 1, 0, x.data_ptr(), dt.data_ptr(), A.data_ptr(),
                   Bm.data_ptr(), Cm.data_ptr(), D.data_ptr(), bias.data_ptr(), 1, None,
                   y.data_ptr(), hl.data_ptr())
    fn, argp = ss.lib().ss_ssd_fwd, ctypes.byref(a)
    sp = ctypes.c_void_p(stream.cuda_stream)
    steps = max(args.steps, 1)

    def timed(handle):
        for _ in range(max(args.warmup, 3)):
            assert fn(handle, argp, sp) == 0
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn(handle, argp, sp)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) * 1e3 / steps

    # the warp-level mma.sync kernel on the same call, for comparison
    mma_ctx = ss.Context(dev.index if dev.index is not None else 0)
    mma_ctx.set_option(ss.SS_OPT_SSD_PATH, ss.SS_SSD_PATH_MMA_SYNC)
    us_mma = timed(mma_ctx.handle)
    mma_ctx.close()
    us = timed(ctx.handle)
    path = "tensor memory (tcgen05)" if ctx.last_launch()[0] == 1 else "mma.sync"
    Q = 64
    chunks = batch * H * (L // Q)
    # per chunk and head: C B^T (2 Q Q N), masked products with x (2 Q Q P),
    # C H_prev^T (2 Q P N), B^T x~ (2 N P Q)
    flops = chunks * (2 * Q * Q * N + 2 * Q * Q * P + 2 * Q * P * N + 2 * N * P * Q)
    tflops = flops / (us * 1e-6) / 1e12
    nbytes = batch * L * (H * P * 2 + H * P * 4 + H * 2 + 2 * N * 2) + 2 * batch * H * P * N * 4
    peak_t = None
    try:
        peak_t = float(json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"])
    except Exception:
        peak_t = 1800.0
    hbm, src = measured_peaks()
    legacy = None
    m = (probes or {}).get("mma_sync_bf16")
    if path == "mma.sync" and m and m.get("rc") == 0 and m.get("sm_ghz", 0) > 0:
        # what mma.sync (the tensor-core path this kernel uses) sustains, at the maximum clock
        lp = m["ops_per_s"] * (MAX_SM_MHZ * 1e-3) / m["sm_ghz"] / 1e12
        legacy = {"peak_tflops": lp, "frac": tflops / lp,
                  "note": "mma.sync m16n8k16 bf16 probe, independent accumulators, 64 warps/SM"}
    return {"workload": "ssd (Mamba-2): batch %d, L %d, %d heads x %d, d_state %d, bf16 in, "
                        "fp32 y" % (batch, L, H, P, N),
            "flops_counted_at_chunk": Q,
            "kernel": path, "us_per_call": us, "mma_sync_kernel_us_per_call": us_mma,
            "elements_per_s": batch * L * H * P / (us * 1e-6),
            "tensor": {"achieved_tflops": tflops, "peak_tflops": peak_t,
                       "frac": tflops / peak_t, "note": "algorithmic bf16 products (the state's "
                       "low bf16 half in C H_prev adds 2 Q P N per chunk, not counted)",
                       "legacy_mma": legacy},
            "hbm": {"gbs": nbytes / (us * 1e-6) / 1e9, "peak": hbm, "peak_source": src,
                    "frac": nbytes / (us * 1e-6) / 1e9 / hbm},
            "steps": steps, "gpu_launches": steps}


def sms_of(dev):
    import torch
    return torch.cuda.get_device_properties(dev).multi_processor_count


def scan_roofline(cfg, avg_s, probes, sms):
    """Roofline of one ss_scan_fwd call on `cfg` taking `avg_s` seconds: the
    HBM, FP32 and ex2 floors (max of them binds), plus the informative issue and
    mixed-unit floors."""
    hbm_peak, hbm_src = measured_peaks()
    nbytes = step_bytes(cfg)
    elements = cfg.elements
    gbs = nbytes / avg_s / 1e9
    bdln = elements * cfg.dstate
    terms = {"hbm": {"achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "peak_source": hbm_src,
                     "floor_us": nbytes / (hbm_peak * 1e9) * 1e6,
                     "frac_of_nominal_8000": gbs / 8000.0}}
    fp32_peak = sms * FP32_LANES_PER_SM * MAX_SM_MHZ * 1e6 / 1e12     # Tops/s
    fp32_ops = 4.0 * bdln
    terms["fp32"] = {"achieved": fp32_ops / avg_s / 1e12, "peak": fp32_peak,
                     "unit": "Tops/s", "floor_us": fp32_ops / (fp32_peak * 1e12) * 1e6,
                     "note": "4 FMA-pipe lane ops per state element (dt*A, dt*u*B, state FMA, "
                             "output FMA) against %d lanes/SM at %.0f MHz" % (FP32_LANES_PER_SM,
                                                                             MAX_SM_MHZ)}
    if probes and probes["ex2"]["rc"] == 0 and probes["ex2"]["sm_ghz"] > 0:
        per_clk = probes["ex2"]["ops_per_s"] / (sms * probes["ex2"]["sm_ghz"] * 1e9)
        per_clk_arch = float(2 ** round(np.log2(max(per_clk, 1e-9))))
        ex2_peak = sms * per_clk_arch * MAX_SM_MHZ * 1e6 / 1e9            # Gex2/s
        # all MUFU work of the call: the N decays per element plus softplus (2) and
        # the gate (2) per (b, d, l)
        mufu_all = elements * (cfg.dstate + 4)
        terms["ex2"] = {"achieved": bdln / avg_s / 1e9, "peak": ex2_peak,
                        "unit": "Gex2/s", "floor_us": bdln / (ex2_peak * 1e9) * 1e6,
                        "ex2_per_clk_per_sm_measured": per_clk,
                        "ex2_per_clk_per_sm_used": per_clk_arch,
                        "mufu_all_ops": mufu_all,
                        "mufu_all_floor_us": mufu_all / (ex2_peak * 1e9) * 1e6}
    for t in terms.values():
        t["frac"] = t["achieved"] / t["peak"]
    dominant = max(terms, key=lambda k: terms[k]["floor_us"])
    # informative: the 4 FP32 lane-ops and the ex2 of a state element all take
    # issue slots of the same warp scheduler (1 warp-instruction per clock per
    # scheduler, 4 schedulers per SM), so 5 slots per 32 elements bound the
    # arithmetic before any overhead; not part of the max above
    issue_floor_us = bdln * 5 / 32 / (4 * sms) / (MAX_SM_MHZ * 1e6) * 1e6
    issue_term = {"floor_us": issue_floor_us, "frac": issue_floor_us / (avg_s * 1e6),
                  "note": "5 issue slots (4 FP32 + 1 MUFU) per 32 state elements, 4 schedulers/SM"}
    # informative: the mixed probe runs ex2 and FFMA2 at the scan's ratio (one
    # ex2 per four FMA lane-ops) on independent chains; its rate, scaled to the
    # maximum clock, is what the two units deliver together
    mixed_term = None
    if probes and probes.get("mixed", {}).get("rc") == 0 and probes["mixed"]["sm_ghz"] > 0:
        rate = probes["mixed"]["ops_per_s"] * (MAX_SM_MHZ * 1e-3) / probes["mixed"]["sm_ghz"]
        per_clk = probes["mixed"]["ops_per_s"] / (sms * probes["mixed"]["sm_ghz"] * 1e9)
        mixed_term = {"floor_us": bdln / rate * 1e6, "frac": bdln / rate / avg_s,
                      "elements_per_clk_per_sm": per_clk,
                      "note": "state elements (1 ex2 + 4 FMA lane-ops) per second that the "
                              "mixed probe sustains, at the maximum clock"}
    dt = terms[dominant]
    floor = max(t["floor_us"] for t in terms.values())
    return {"bound": "hbm" if dominant == "hbm" else "alu", "term": dominant,
            "achieved": dt["achieved"], "peak": dt["peak"], "unit": dt["unit"],
            "frac": dt["frac"], "traffic": None, "algorithmic_bytes_per_launch": nbytes,
            "kernel_us": avg_s * 1e6, "floor_us": floor, "frac_of_floor": floor / (avg_s * 1e6),
            "terms": terms, "issue_slots": issue_term, "mixed_units": mixed_term,
            "peak_clock_mhz": MAX_SM_MHZ}


def time_scan_config(ss, ctx, dev, stream, name, probes, warmup=3, steps=10):
    """One other configuration of the scan (its own inputs, resident): time per
    call from CUDA events on the launching stream, elements/s and its roofline."""
    import torch
    cfg = workloads.CONFIGS[name]
    inp = workloads.scan_inputs(cfg)
    shp = (cfg.batch, cfg.dim, cfg.seqlen)

    def to_dev(a, shape):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).reshape(shape).to(dev)
        return torch.from_numpy(a).reshape(shape).to(dev)

    t = {k: to_dev(inp[k], shp) for k in ("u", "delta", "z")}
    t["B"] = to_dev(inp["B"], inp["B"].shape)
    t["C"] = to_dev(inp["C"], inp["C"].shape)
    prm = {k: torch.from_numpy(inp[k]).to(dev) for k in ("A", "D", "delta_bias")}
    del inp
    y = torch.empty(shp, dtype=torch.float32, device=dev)
    hl = torch.empty((cfg.batch, cfg.dim, cfg.dstate), dtype=torch.float32, device=dev)
    call = ss.PreparedScan(t["u"], t["delta"], prm["A"], t["B"], t["C"], D=prm["D"],
                           delta_bias=prm["delta_bias"], z=t["z"], y=y, h_last=hl, ctx=ctx,
                           stream=stream)
    if cfg.seqlen > 100000:
        steps = max(3, steps // 2)
    for _ in range(warmup):
        call()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    if ctx.device_error() != ss.SS_OK:
        raise RuntimeError("device error in the %s leg" % name)
    variant, launches = ctx.last_launch()
    avg_s = e0.elapsed_time(e1) / steps * 1e-3
    rf = scan_roofline(cfg, avg_s, probes, sms_of(dev))
    names = {0: "auto", 1: "rows", 2: "chunked", 3: "simple"}
    return {"workload": workload_config(cfg)["workload"], "us_per_call": avg_s * 1e6,
            "elements_per_s": cfg.elements / avg_s, "gbs": rf["terms"]["hbm"]["achieved"],
            "variant": names.get(variant, str(variant)), "launches_per_call": launches,
            "roofline": {k: rf[k] for k in ("bound", "term", "achieved", "peak", "unit", "frac",
                                            "floor_us", "frac_of_floor", "terms")},
            "steps": steps, "gpu_launches": steps * launches}


def run_ours(args, rank, world, local):
    import torch
    import selective_state_space_136_b300 as ss

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    cfg = workloads.CONFIGS[args.config]
    inp = workloads.scan_inputs(cfg)
    shp = (cfg.batch, cfg.dim, cfg.seqlen)

    def host_tensor(a, shape):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).reshape(shape)
        return torch.from_numpy(a).reshape(shape)

    host = {k: host_tensor(inp[k], shp) for k in ("u", "delta", "z")}
    host["B"] = host_tensor(inp["B"], inp["B"].shape)
    host["C"] = host_tensor(inp["C"], inp["C"].shape)
    params = {k: torch.from_numpy(inp[k]).to(dev) for k in ("A", "D", "delta_bias")}
    d = {k: v.to(dev) for k, v in host.items()}
    y = torch.empty(shp, dtype=torch.float32, device=dev)
    h_last = torch.empty((cfg.batch, cfg.dim, cfg.dstate), dtype=torch.float32, device=dev)

    ctx = ss.Context(local)
    ctx.set_option(ss.SS_OPT_VARIANT, {"auto": 0, "rows": 1, "chunked": 2, "simple": 3}[args.variant])
    ctx.set_option(ss.SS_OPT_THREADS_PER_ROW, args.tpr)
    ctx.set_option(ss.SS_OPT_SEGMENTS, args.segments)
    stream = torch.cuda.current_stream(dev)

    def step(t):
        ss.ss_scan_fwd(t["u"], t["delta"], params["A"], t["B"], t["C"], D=params["D"],
                       delta_bias=params["delta_bias"], z=t["z"], y=y, h_last=h_last, ctx=ctx,
                       stream=stream)

    # the device-resident loop: arguments checked and marshalled once, so the
    # timed region measures the GPU work rather than Python argument checks
    resident_call = ss.PreparedScan(d["u"], d["delta"], params["A"], d["B"], d["C"],
                                    D=params["D"], delta_bias=params["delta_bias"], z=d["z"],
                                    y=y, h_last=h_last, ctx=ctx, stream=stream)

    probes = None if args.skip_probe else probe_alu(local)

    for _ in range(max(args.warmup, 0)):
        resident_call()
    torch.cuda.synchronize(dev)
    if ctx.device_error() != ss.SS_OK:
        raise RuntimeError("device error during warm-up")
    variant, launches_per_step = ctx.last_launch()

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if pg:
        pg.barrier()
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    t_wall0 = time.perf_counter()
    ev[0].record(stream)
    for i in range(args.steps):
        resident_call()
        ev[i + 1].record(stream)
    t_enq = time.perf_counter()
    torch.cuda.synchronize(dev)
    t_wall1 = time.perf_counter()
    if pg:
        pg.barrier()
    clocks = sampler.stop(t_wall0, t_wall1)
    per_launch_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    total_ms = ev[0].elapsed_time(ev[-1])
    if ctx.device_error() != ss.SS_OK:
        raise RuntimeError("device error in the timed region")
    total_ms = max_over_ranks(pg, total_ms, dev)

    elements = cfg.elements
    value = replica_throughput(world, elements, args.steps, total_ms)
    ms_per_step = total_ms / args.steps
    # one call = the whole path (B/C pack + scan); the scan kernel is ~99% of it
    avg_launch_s = float(np.mean(per_launch_ms)) * 1e-3
    host_us_per_call = (t_enq - t_wall0) / args.steps * 1e6

    decode = None if args.skip_decode else time_decode(ss, ctx, dev, stream, args)
    conv1d = None if args.skip_conv else time_conv1d(ss, ctx, dev, stream, cfg, args)
    bwd = None if args.skip_bwd else time_bwd(ss, ctx, dev, stream, cfg, d, params, args)
    conv_scan = None if args.skip_conv else time_conv_scan(ss, ctx, dev, stream, cfg, d, params,
                                                           args, probes)
    ssd = None if args.skip_ssd else time_ssd(ss, ctx, dev, stream, args, probes=probes)

    # ---- end to end: pinned host inputs in, y and h_last back to host, every step.
    # Steps are pipelined over two buffer sets and three streams: the inputs of
    # step k+1 go up while the scan of step k runs and its results come down
    # (PCIe is full duplex). Each step still copies all of its own inputs in and
    # its y and h_last out.
    e2e = None
    if not args.skip_e2e:
        pinned = {k: v.pin_memory() for k, v in host.items()}
        y_host = [torch.empty(shp, dtype=torch.float32).pin_memory() for _ in range(2)]
        h_host = [torch.empty((cfg.batch, cfg.dim, cfg.dstate), dtype=torch.float32).pin_memory()
                  for _ in range(2)]
        h2d = sum(v.numel() * v.element_size() for v in pinned.values())
        d2h = y_host[0].numel() * 4 + h_host[0].numel() * 4
        dd = [{k: torch.empty_like(v) for k, v in d.items()} for _ in range(2)]
        yd = [torch.empty_like(y) for _ in range(2)]
        hd = [torch.empty_like(h_last) for _ in range(2)]
        s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()
        up_done, comp_done, down_done = {}, {}, {}

        def e2e_step(k):
            i = k % 2
            with torch.cuda.stream(s_up):
                if k - 2 in comp_done:  # the scan of step k-2 has read buffer set i
                    s_up.wait_event(comp_done[k - 2])
                for name in dd[i]:
                    dd[i][name].copy_(pinned[name], non_blocking=True)
                up_done[k] = ev()
                up_done[k].record(s_up)
            stream.wait_event(up_done[k])
            if k - 2 in down_done:  # the results of step k-2 have left y/h buffer i
                stream.wait_event(down_done[k - 2])
            t = dd[i]
            ss.ss_scan_fwd(t["u"], t["delta"], params["A"], t["B"], t["C"], D=params["D"],
                           delta_bias=params["delta_bias"], z=t["z"], y=yd[i], h_last=hd[i],
                           ctx=ctx, stream=stream)
            comp_done[k] = ev()
            comp_done[k].record(stream)
            with torch.cuda.stream(s_down):
                s_down.wait_event(comp_done[k])
                y_host[i].copy_(yd[i], non_blocking=True)
                h_host[i].copy_(hd[i], non_blocking=True)
                down_done[k] = ev()
                down_done[k].record(s_down)

        for k in range(2):
            e2e_step(k)
        torch.cuda.synchronize(dev)
        up_done.clear(), comp_done.clear(), down_done.clear()
        k_e2e = max(2, min(args.steps, 8))
        if pg:
            pg.barrier()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for k in range(k_e2e):
            e2e_step(k)
        torch.cuda.synchronize(dev)
        e_ms = (time.perf_counter() - t0) * 1e3
        e_ms = max_over_ranks(pg, e_ms, dev)
        e2e = {"value": replica_throughput(world, elements, k_e2e, e_ms), "unit": "elements/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k_e2e,
               "note": "pinned host buffers; wall clock around the steps with a synchronize on "
                       "both sides; inputs of step k+1 copied in while step k computes and "
                       "copies out"}

    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return

    # ---- roofline of the (single) scan kernel
    roofline = scan_roofline(cfg, avg_launch_s, probes, sms_of(dev))
    roofline["traffic"] = committed_traffic(args.config)
    roofline["kernel_note"] = ("time of one ss_scan_fwd call (B/C pack + scan kernels) from CUDA "
                               "events on the launching stream, averaged over the timed steps")
    nbytes = roofline["algorithmic_bytes_per_launch"]
    gbs = roofline["terms"]["hbm"]["achieved"]

    per_config = None
    if not args.skip_configs:
        per_config = {}
        for name in ("mamba130m", "long1m"):
            if name != args.config:
                per_config[name] = time_scan_config(ss, ctx, dev, stream, name, probes)

    cpu = None
    if not args.skip_cpu:
        cores = cpu_cores()
        v, nrows, distinct, el = time_oracle(cfg, args.cpu_seconds, cores)
        cpu = {"value": v, "unit": "elements/s", "cores": cores, "kind": "oracle",
               "sample": "%d row scans at full L=%d over the first %d of the %d rows (b,d) of %s, "
                         "repeated; %.1f s timed, fp64 C oracle"
                         % (nrows, cfg.seqlen, distinct, cfg.rows, args.config, el)}

    names = {0: "auto", 1: "rows", 2: "chunked", 3: "simple"}
    out = {
        "metric": METRIC, "value": value, "unit": "elements/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded normal draws; A=-(n+1); dt bias log-uniform [1e-3,1e-1])",
        "config": dict(workload_config(cfg),
                       parallelism="replicas" if world > 1 else "single"),
        "variant": names.get(variant, str(variant)),
        "l2": "no flush: %.0f MB of inputs+outputs per step > 126 MB L2" % (nbytes / 1e6),
        "gbs": gbs,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clocks,
        "gpu_launches": int(args.steps * launches_per_step),
        "host_us_per_call": host_us_per_call,
        "alu_probe": probes,
        "decode": decode,
        "conv1d": conv1d,
        "conv_scan": conv_scan,
        "backward": bwd,
        "ssd": ssd,
        "configs": per_config,
        "impl": "ours",
    }
    print(json.dumps(out), flush=True)
    if pg:
        pg.destroy_process_group()


# ---------------------------------------------------------------- reference arm (the oracle)

def run_reference(args, rank, world):
    if rank != 0:
        return
    cfg = workloads.CONFIGS[args.config]
    cores = cpu_cores()
    per_step = max(1.0, min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        time_oracle(cfg, per_step / 4, cores)
    vals, rows_done, secs, distinct = [], 0, 0.0, 0
    for _ in range(args.steps):
        v, nrows, distinct, el = time_oracle(cfg, per_step, cores)
        vals.append(v)
        rows_done += nrows
        secs += el
    value = float(np.mean(vals))
    sample = ("%d row scans at full L=%d over the first %d of the %d rows (b,d) of %s, repeated, "
              "in %d steps; %.1f s timed, fp64 C oracle on %d host threads"
              % (rows_done, cfg.seqlen, distinct, cfg.rows, args.config, args.steps, secs, cores))
    out = {"metric": METRIC, "value": value, "unit": "elements/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": cfg.elements / value * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": dict(workload_config(cfg),
                          parallelism="replicas" if world > 1 else "single"),
           "impl": "reference",
           "cpu_baseline": {"value": value, "unit": "elements/s", "cores": cores,
                            "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "elements/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0},
           "gpu_launches": 0}
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
