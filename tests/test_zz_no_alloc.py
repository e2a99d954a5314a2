"""ss_scan_fwd_noalloc: the allocation-free entry point (through the C ABI).

It serves callers that may not call cudaMalloc (memory-planned or captured
regions, allocator-free real-time paths, host-owned-memory plugins): its
scratch is a static device array of the library. Its output must match the
regular entry point's on the same inputs, call after call, and shapes whose
scratch would not fit are refused before anything is enqueued.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from gpu_util import check_close, device_inputs, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu

ss = pytest.importorskip("selective_state_space_136_b300")


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = ss.lib()
    L.ss_scan_fwd_noalloc.argtypes = [ctypes.POINTER(ss.ScanArgs), ctypes.c_void_p, ctypes.c_void_p]
    L.ss_scan_fwd_noalloc.restype = ctypes.c_int
    return L


def _args(cfg, t, y, hl):
    return ss.ScanArgs(cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen, ss.SS_BF16, ss.SS_F32,
                       t["u"].data_ptr(), t["delta"].data_ptr(), t["z"].data_ptr(),
                       t["A"].data_ptr(), t["B"].data_ptr(), t["C"].data_ptr(),
                       t["D"].data_ptr(), t["delta_bias"].data_ptr(), 1, None,
                       y.data_ptr(), hl.data_ptr())


def test_matches_regular_entry_point_twice(lib):
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    for seed in (71, 72):  # two calls in a row: the second reuses the stale scratch
        cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=2, dim=96, seqlen=512,
                               seed=seed)
        t = device_inputs(workloads.scan_inputs(cfg), cfg)
        y_ref, h_ref = ss.ss_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"],
                                      delta_bias=t["delta_bias"], z=t["z"])
        y = torch.full_like(y_ref, float("nan"))
        hl = torch.full_like(h_ref, float("nan"))
        a = _args(cfg, t, y, hl)
        assert lib.ss_scan_fwd_noalloc(ctypes.byref(a), ctypes.c_void_p(err.data_ptr()), st) == 0
        torch.cuda.synchronize()
        assert int(err[0].item()) == 0
        check_close(y.cpu().numpy(), y_ref.cpu().numpy(), True, "y")
        check_close(hl.cpu().numpy(), h_ref.cpu().numpy(), True, "h_last")


def test_split_row_blocks_twice_against_oracle(lib):
    """More row blocks (2048) than chained ranges (8 per SM), so row blocks are
    split between two ranges and their tail pieces wait on flags in the shared
    array; the second call must ignore the first call's flags and carries."""
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    err = torch.zeros(4, dtype=torch.int32, device="cuda")
    for seed in (81, 82):
        cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=8, dim=8192, seqlen=64,
                               seed=seed)
        inp = workloads.scan_inputs(cfg)
        t = device_inputs(inp, cfg)
        y_ref, h_ref = ss.ss_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"],
                                      delta_bias=t["delta_bias"], z=t["z"])
        y = torch.full_like(y_ref, float("nan"))
        hl = torch.full_like(h_ref, float("nan"))
        assert lib.ss_scan_fwd_noalloc(ctypes.byref(_args(cfg, t, y, hl)),
                                       ctypes.c_void_p(err.data_ptr()), st) == 0
        torch.cuda.synchronize()
        assert int(err[0].item()) == 0
        check_close(y.cpu().numpy(), y_ref.cpu().numpy(), True, "y vs ss_scan_fwd")
        check_close(hl.cpu().numpy(), h_ref.cpu().numpy(), True, "h_last vs ss_scan_fwd")
        rows = sample_rows(cfg, 64, seed=seed)
        yo, ho = oracle_rows(inp, cfg, rows)
        yg = y.reshape(cfg.rows, cfg.seqlen).cpu().numpy()[rows]
        hg = hl.reshape(cfg.rows, cfg.dstate).cpu().numpy()[rows]
        check_close(yg, yo, True, "y vs oracle")
        check_close(hg, ho, True, "h_last vs oracle")


def test_refuses_shapes_beyond_the_static_scratch(lib):
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # seqlen 65536: the packed B/C alone would take the whole 8 MiB
    big = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=1, dim=32, seqlen=65536)
    shp = (big.batch, big.dim, big.seqlen)
    bf = torch.bfloat16
    t = {k: torch.zeros(shp, dtype=bf, device="cuda") for k in ("u", "delta", "z")}
    t["B"] = torch.zeros(big.batch, big.dstate, big.seqlen, dtype=bf, device="cuda")
    t["C"] = torch.zeros_like(t["B"])
    t["A"] = -torch.ones(big.dim, big.dstate, device="cuda")
    t["D"] = torch.zeros(big.dim, device="cuda")
    t["delta_bias"] = torch.zeros(big.dim, device="cuda")
    y = torch.full(shp, 5.0, device="cuda")
    hl = torch.empty(big.batch, big.dim, big.dstate, device="cuda")
    assert lib.ss_scan_fwd_noalloc(ctypes.byref(_args(big, t, y, hl)), None, st) == \
        ss.SS_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((y == 5.0).all())  # nothing was enqueued
    # shapes the entry point does not serve
    small = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=1, dim=32, seqlen=16)
    ts = device_inputs(workloads.scan_inputs(small), small)
    ys = torch.empty(small.batch, small.dim, small.seqlen, device="cuda")
    hs = torch.empty(small.batch, small.dim, small.dstate, device="cuda")
    a = _args(small, ts, ys, hs)
    a.dstate = 4
    assert lib.ss_scan_fwd_noalloc(ctypes.byref(a), None, st) == ss.SS_ERR_UNSUPPORTED
    assert lib.ss_scan_fwd_noalloc(None, None, st) == ss.SS_ERR_INVALID_ARG
