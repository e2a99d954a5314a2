"""GPU parity of ss_scan_fwd against the fp64 oracle (through the C ABI)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import (check_close, dev_tensor, device_inputs, oracle_rows, sample_rows)

pytestmark = pytest.mark.gpu

ss = pytest.importorskip("selective_state_space_136_b300")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.init()


def _ctx(variant=ss.SS_VARIANT_AUTO, tpr=0, segments=0):
    c = ss.Context(0)
    c.set_option(ss.SS_OPT_VARIANT, variant)
    c.set_option(ss.SS_OPT_THREADS_PER_ROW, tpr)
    c.set_option(ss.SS_OPT_SEGMENTS, segments)
    return c


def _run(cfg, t, ctx, with_z=True, with_D=True, with_bias=True, softplus=True, h0=None,
         out_dtype=torch.float32):
    y, hl = ss.ss_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"],
                           D=t["D"] if with_D else None,
                           delta_bias=t["delta_bias"] if with_bias else None,
                           z=t["z"] if with_z else None, delta_softplus=softplus, h0=h0,
                           out_dtype=out_dtype, ctx=ctx)
    torch.cuda.synchronize()
    assert ctx.device_error() == ss.SS_OK
    return y.float().cpu().numpy().astype(np.float64), hl.cpu().numpy().astype(np.float64)


def _full_check(cfg, variant, tpr=0, out_dtype=torch.float32, with_h0=False, **flags):
    inp = workloads.scan_inputs(cfg, with_h0=with_h0)
    t = device_inputs(inp, cfg)
    ctx = _ctx(variant, tpr)
    y, hl = _run(cfg, t, ctx, h0=t.get("h0"), out_dtype=out_dtype, **flags)
    rows = np.arange(cfg.rows)
    y_ref, h_ref = oracle_rows(inp, cfg, rows, h0=inp.get("h0"), **flags)
    bf = cfg.in_dtype == "bf16" or out_dtype == torch.bfloat16
    check_close(y.reshape(cfg.rows, cfg.seqlen), y_ref, bf, "y")
    check_close(hl.reshape(cfg.rows, cfg.dstate), h_ref, cfg.in_dtype == "bf16", "h_last")
    return ctx


# ---------------------------------------------------------------- small and edge shapes

def test_tiny_config_rows_and_simple():
    cfg = workloads.CONFIGS["tiny"]
    for v in (ss.SS_VARIANT_AUTO, ss.SS_VARIANT_ROWS, ss.SS_VARIANT_SIMPLE):
        ctx = _full_check(cfg, v)
        want = ss.SS_VARIANT_SIMPLE if v == ss.SS_VARIANT_SIMPLE else ss.SS_VARIANT_ROWS
        assert ctx.last_launch() == (want, 1)


EDGE = [
    # (N, L, dim, batch, in_dtype)
    (16, 64, 64, 2, "bf16"),
    (16, 72, 33, 3, "bf16"),      # dim not a multiple of the CTA rows, ragged tile
    (16, 1032, 40, 1, "bf16"),
    (16, 8, 32, 1, "f32"),
    (16, 96, 70, 2, "f32"),
    (8, 136, 65, 2, "bf16"),
    (4, 40, 129, 1, "bf16"),
    (2, 48, 17, 2, "f32"),
    (1, 200, 5, 2, "bf16"),
    (16, 1, 24, 2, "bf16"),       # L = 1 (simple path)
    (16, 7, 24, 2, "f32"),        # L not a multiple of 8 (simple path)
    (16, 63, 24, 1, "bf16"),
    (16, 65, 24, 1, "bf16"),
    (4, 129, 9, 1, "f32"),
]


@pytest.mark.parametrize("N,L,dim,batch,dt", EDGE)
def test_edge_shapes(N, L, dim, batch, dt):
    cfg = workloads.scaled(workloads.CONFIGS["mamba130m"], batch=batch, dim=dim, dstate=N,
                           seqlen=L, in_dtype=dt, seed=40 + N + L)
    variants = [ss.SS_VARIANT_AUTO, ss.SS_VARIANT_SIMPLE]
    for v in variants:
        _full_check(cfg, v)


@pytest.mark.parametrize("flags", [
    dict(with_z=False), dict(with_D=False), dict(with_bias=False), dict(softplus=False),
    dict(with_z=False, with_D=False, with_bias=False)])
@pytest.mark.parametrize("variant", ["AUTO", "SIMPLE"])
def test_optional_inputs(flags, variant):
    cfg = workloads.scaled(workloads.CONFIGS["mamba130m"], batch=2, dim=48, seqlen=256, seed=51)
    if flags.get("softplus") is False:
        # keep dt = delta + bias positive and moderate when used as is
        cfg = workloads.scaled(cfg, seed=52)
    inp = workloads.scan_inputs(cfg)
    if flags.get("softplus") is False:
        inp["delta"] = workloads.f32_to_bf16_bits(
            np.abs(workloads.bf16_bits_to_f32(inp["delta"])) * 0.05)
        inp["delta_bias"] = np.abs(inp["delta_bias"]) * 0.0 + 0.01
    t = device_inputs(inp, cfg)
    ctx = _ctx(getattr(ss, "SS_VARIANT_" + variant))
    y, hl = _run(cfg, t, ctx, **flags)
    y_ref, h_ref = oracle_rows(inp, cfg, np.arange(cfg.rows), **flags)
    check_close(y.reshape(cfg.rows, -1), y_ref, True, "y")
    check_close(hl.reshape(cfg.rows, -1), h_ref, True, "h_last")


@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_initial_state_and_bf16_output(dt):
    cfg = workloads.scaled(workloads.CONFIGS["mamba130m"], batch=2, dim=40, seqlen=128,
                           in_dtype=dt, seed=53)
    _full_check(cfg, ss.SS_VARIANT_AUTO, with_h0=True)
    _full_check(cfg, ss.SS_VARIANT_AUTO, out_dtype=torch.bfloat16)
    _full_check(cfg, ss.SS_VARIANT_SIMPLE, with_h0=True, out_dtype=torch.bfloat16)


@pytest.mark.parametrize("tpr", [1, 2, 4])
def test_threads_per_row(tpr):
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=2, dim=96, seqlen=528, seed=54)
    _full_check(cfg, ss.SS_VARIANT_ROWS, tpr=tpr)


@pytest.mark.parametrize("batch,dim,seqlen,warps_per_sm,dt", [
    (3, 3200, 160, 1, "f32"),    # ~2 row blocks per warp: tail, whole block, head
    (3, 3200, 160, 2, "bf16"),   # barely more row blocks than warps: tiny slack
    (2, 4736, 160, 2, "f32"),    # exactly one row block per warp
    (2, 4736, 528, 1, "bf16"),   # exactly two per warp, odd tile count
    (3, 3190, 160, 1, "f32"),    # partial last row block of each batch
    (1, 640, 160, 1, "f32"),     # fewer row blocks than warps
])
def test_chained_wraparound(batch, dim, seqlen, warps_per_sm, dt):
    """The chained kernel cuts the row blocks' tiles, laid end to end, into
    one equal range per warp; a row block split between two ranges passes its
    state from its head piece to its tail piece through the carry buffer. Every
    output and final state matches the oracle, with and without h0."""
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=batch, dim=dim, seqlen=seqlen,
                           in_dtype=dt, seed=59 + dim % 97 + warps_per_sm)
    inp = workloads.scan_inputs(cfg, with_h0=True)
    t = device_inputs(inp, cfg)
    ctx = _ctx(ss.SS_VARIANT_ROWS, 2)
    ctx.set_option(ss.SS_OPT_RESIDENT_WARPS, warps_per_sm)
    for h0 in (t["h0"], None):
        y, hl = _run(cfg, t, ctx, h0=h0)
        assert ctx.last_launch() == (ss.SS_VARIANT_ROWS, 2)
        y_ref, h_ref = oracle_rows(inp, cfg, np.arange(cfg.rows),
                                   h0=inp["h0"] if h0 is not None else None)
        check_close(y.reshape(cfg.rows, -1), y_ref, dt == "bf16", "y")
        check_close(hl.reshape(cfg.rows, -1), h_ref, dt == "bf16", "h_last")


@pytest.mark.parametrize("segments,dt,dim", [(2, "bf16", 64), (3, "f32", 70), (33, "bf16", 33),
                                             (40, "bf16", 96), (0, "bf16", 160)])
def test_chunked_variant(segments, dt, dim):
    """Segments scanned in parallel, carries combined by the shuffle scan,
    segments re-scanned: same answer as the oracle for any segment count
    (33 and 40 need two combine rounds of 32 segments)."""
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=2, dim=dim, seqlen=640,
                           in_dtype=dt, seed=61 + segments)
    inp = workloads.scan_inputs(cfg, with_h0=True)
    t = device_inputs(inp, cfg)
    ctx = _ctx(ss.SS_VARIANT_CHUNKED, 0, segments)
    for h0 in (t["h0"], None):
        y, hl = _run(cfg, t, ctx, h0=h0)
        assert ctx.last_launch()[0] == ss.SS_VARIANT_CHUNKED
        y_ref, h_ref = oracle_rows(inp, cfg, np.arange(cfg.rows),
                                   h0=inp["h0"] if h0 is not None else None)
        check_close(y.reshape(cfg.rows, -1), y_ref, dt == "bf16", "y")
        check_close(hl.reshape(cfg.rows, -1), h_ref, dt == "bf16", "h_last")


def test_chunked_long_memory():
    """Tiny time steps (bias -> dt ~ 1e-5): the state carries across every
    segment boundary, so a wrong carry shows up at once."""
    cfg = workloads.scaled(workloads.CONFIGS["long1m"], batch=1, dim=64, seqlen=4096, seed=62,
                           dt_lo=1e-5, dt_hi=1e-4)
    inp = workloads.scan_inputs(cfg)
    t = device_inputs(inp, cfg)
    y, hl = _run(cfg, t, _ctx(ss.SS_VARIANT_CHUNKED, 0, 16))
    y_ref, h_ref = oracle_rows(inp, cfg, np.arange(cfg.rows))
    check_close(y.reshape(cfg.rows, -1), y_ref, True, "y")
    check_close(hl.reshape(cfg.rows, -1), h_ref, True, "h_last")


def test_chained_kernel_needs_whole_tiles():
    """seqlen not a multiple of 16: the forced chained variant reports
    unsupported; the automatic choice falls back and stays correct."""
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=1, dim=64, seqlen=520, seed=60)
    inp = workloads.scan_inputs(cfg)
    t = device_inputs(inp, cfg)
    with pytest.raises(ss.SSError) as ei:
        _run(cfg, t, _ctx(ss.SS_VARIANT_ROWS, 2))
    assert ei.value.status == ss.SS_ERR_UNSUPPORTED
    _full_check(cfg, ss.SS_VARIANT_AUTO)


def test_prepared_call_matches():
    """A PreparedScan re-enqueues exactly the call ss_scan_fwd makes."""
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=2, dim=96, seqlen=256, seed=63)
    inp = workloads.scan_inputs(cfg, with_h0=True)
    t = device_inputs(inp, cfg)
    ctx = _ctx()
    y0, h0_ = _run(cfg, t, ctx, h0=t["h0"])
    call = ss.PreparedScan(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"],
                           delta_bias=t["delta_bias"], z=t["z"], h0=t["h0"],
                           h_last=torch.empty_like(t["h0"]), ctx=ctx)
    for _ in range(2):
        y, hl = call()
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy().astype(np.float64), y0)
        assert np.array_equal(hl.cpu().numpy().astype(np.float64), h0_)


def test_moderate_full_tensor():
    """Every element of a multi-tile, multi-CTA case."""
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=2, dim=160, seqlen=1024, seed=55)
    _full_check(cfg, ss.SS_VARIANT_AUTO)


def test_every_output_written_and_no_spill():
    """NaN-poisoned outputs come back finite; guard words around y and h_last
    keep their values."""
    cfg = workloads.scaled(workloads.CONFIGS["mamba130m"], batch=2, dim=36, seqlen=200, seed=56)
    inp = workloads.scan_inputs(cfg)
    t = device_inputs(inp, cfg)
    for v in (ss.SS_VARIANT_AUTO, ss.SS_VARIANT_SIMPLE):
        n_y, n_h, pad = cfg.rows * cfg.seqlen, cfg.rows * cfg.dstate, 64
        ybuf = torch.full((n_y + 2 * pad,), float("nan"), device="cuda")
        hbuf = torch.full((n_h + 2 * pad,), float("nan"), device="cuda")
        ybuf[:pad] = 7.0
        ybuf[-pad:] = 7.0
        hbuf[:pad] = 7.0
        hbuf[-pad:] = 7.0
        y = ybuf[pad:pad + n_y].view(cfg.batch, cfg.dim, cfg.seqlen)
        hl = hbuf[pad:pad + n_h].view(cfg.batch, cfg.dim, cfg.dstate)
        ctx = _ctx(v)
        ss.ss_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"],
                       delta_bias=t["delta_bias"], z=t["z"], y=y, h_last=hl, ctx=ctx)
        torch.cuda.synchronize()
        assert torch.isfinite(y).all() and torch.isfinite(hl).all()
        assert (ybuf[:pad] == 7).all() and (ybuf[-pad:] == 7).all()
        assert (hbuf[:pad] == 7).all() and (hbuf[-pad:] == 7).all()
        y_ref, h_ref = oracle_rows(inp, cfg, np.arange(cfg.rows))
        check_close(y.cpu().numpy().reshape(cfg.rows, -1), y_ref, True, "y")


def test_chunk_split_on_gpu():
    """[0, L) in one call equals [0, L1) then [L1, L) resumed from h_{L1}."""
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=2, dim=64, seqlen=512, seed=57)
    inp = workloads.scan_inputs(cfg)
    t = device_inputs(inp, cfg)
    ctx = _ctx()
    y, hl = _run(cfg, t, ctx)
    L1 = 200
    part = lambda k, s: t[k][..., s].contiguous()
    t1 = dict(t, **{k: part(k, slice(0, L1)) for k in ("u", "delta", "z", "B", "C")})
    t2 = dict(t, **{k: part(k, slice(L1, None)) for k in ("u", "delta", "z", "B", "C")})
    y1, h1 = _run(cfg, t1, ctx)
    y2, h2 = _run(cfg, t2, ctx, h0=torch.from_numpy(h1.astype(np.float32)).cuda())
    y_ref, h_ref = oracle_rows(inp, cfg, np.arange(cfg.rows))
    check_close(np.concatenate([y1, y2], axis=-1).reshape(cfg.rows, -1), y_ref, True, "split y")
    check_close(h2.reshape(cfg.rows, -1), h_ref, True, "split h")
    assert np.max(np.abs(np.concatenate([y1, y2], axis=-1) - y)) <= 1e-4 * np.max(np.abs(y))


def test_zero_length_sequence():
    cfg = workloads.scaled(workloads.CONFIGS["tiny"], seqlen=8)
    inp = workloads.scan_inputs(cfg, with_h0=True)
    t = device_inputs(inp, cfg)
    e = lambda k: t[k][..., :0].contiguous()
    hl = torch.full_like(t["h0"], float("nan"))
    y, hl = ss.ss_scan_fwd(e("u"), e("delta"), t["A"], e("B"), e("C"), D=t["D"], z=e("z"),
                           h0=t["h0"], h_last=hl)
    torch.cuda.synchronize()
    assert y.numel() == 0 and torch.equal(hl, t["h0"])


# ---------------------------------------------------------------- full-size configs

def _config_sampled(name, n_rows, variant=ss.SS_VARIANT_AUTO):
    cfg = workloads.CONFIGS[name]
    inp = workloads.scan_inputs(cfg)
    t = device_inputs(inp, cfg)
    ctx = _ctx(variant)
    y, hl = ss.ss_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"],
                           delta_bias=t["delta_bias"], z=t["z"], ctx=ctx)
    torch.cuda.synchronize()
    assert ctx.device_error() == ss.SS_OK
    rows = sample_rows(cfg, n_rows)
    y_ref, h_ref = oracle_rows(inp, cfg, rows)
    yv = y.view(cfg.rows, cfg.seqlen)[torch.from_numpy(rows).cuda()].cpu().numpy()
    hv = hl.view(cfg.rows, cfg.dstate)[torch.from_numpy(rows).cuda()].cpu().numpy()
    check_close(yv, y_ref, True, name + " y")
    check_close(hv, h_ref, True, name + " h_last")
    return ctx


def test_config_mamba130m_sampled():
    _config_sampled("mamba130m", 256)


def test_config_mamba2p8b_sampled():
    """The benchmark's workload and launch configuration."""
    _config_sampled("mamba2p8b", 256)


def test_config_long1m_sampled():
    """64 seeded rows (plus the edge rows) of the 1536 over the full L = 2^20."""
    _config_sampled("long1m", 64)


# ---------------------------------------------------------------- host checks and device waits

def test_host_rejects_bad_arguments():
    cfg = workloads.scaled(workloads.CONFIGS["tiny"], seqlen=16)
    t = device_inputs(workloads.scan_inputs(cfg), cfg)
    ctx = _ctx()
    a = ss.ScanArgs(cfg.batch, cfg.dim, cfg.dstate, cfg.seqlen, ss.SS_F32, ss.SS_F32,
                    t["u"].data_ptr(), t["delta"].data_ptr(), None, t["A"].data_ptr(),
                    t["B"].data_ptr(), t["C"].data_ptr(), None, None, 1, None, None, None)
    y = torch.empty_like(t["u"])
    a.y = y.data_ptr()
    L = ss.lib()
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert L.ss_scan_fwd(ctx.handle, ctypes.byref(a), st) == ss.SS_OK
    bad = ss.ScanArgs.from_buffer_copy(a)
    bad.u = t["u"].data_ptr() + 4                       # misaligned
    assert L.ss_scan_fwd(ctx.handle, ctypes.byref(bad), st) == ss.SS_ERR_INVALID_ARG
    bad = ss.ScanArgs.from_buffer_copy(a)
    bad.y = t["u"].data_ptr()                           # output aliases an input
    assert L.ss_scan_fwd(ctx.handle, ctypes.byref(bad), st) == ss.SS_ERR_INVALID_ARG
    bad = ss.ScanArgs.from_buffer_copy(a)
    bad.dstate = 3
    assert L.ss_scan_fwd(ctx.handle, ctypes.byref(bad), st) == ss.SS_ERR_UNSUPPORTED
    bad = ss.ScanArgs.from_buffer_copy(a)
    bad.in_dtype = 7
    assert L.ss_scan_fwd(ctx.handle, ctypes.byref(bad), st) == ss.SS_ERR_INVALID_ARG
    torch.cuda.synchronize()


@pytest.mark.parametrize("tpr", [1, 2, 4, "chunked"])
@pytest.mark.parametrize("drop", [0, 3])
def test_device_wait_times_out_cleanly(tpr, drop):
    """A tile whose loads are never issued makes the bounded wait run out: the
    kernel records SS_ERR_TIMEOUT and returns; the context keeps working."""
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=1, dim=64, seqlen=256, seed=58)
    inp = workloads.scan_inputs(cfg)
    t = device_inputs(inp, cfg)
    if tpr == "chunked":
        ctx = _ctx(ss.SS_VARIANT_CHUNKED, 0, 2)
    else:
        ctx = _ctx(ss.SS_VARIANT_ROWS, tpr)
    ctx.set_option(ss.SS_OPT_WAIT_LIMIT, 2000)
    ctx.set_option(ss.SS_OPT_TEST_DROP_TILE, drop)
    ss.ss_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"],
                   delta_bias=t["delta_bias"], z=t["z"], ctx=ctx)
    assert ctx.device_error() == ss.SS_ERR_TIMEOUT
    assert ctx.device_error() == ss.SS_OK  # cleared by the read
    ctx.set_option(ss.SS_OPT_TEST_DROP_TILE, -1)
    ctx.set_option(ss.SS_OPT_WAIT_LIMIT, 1 << 22)
    y, hl = _run(cfg, t, ctx)
    y_ref, _ = oracle_rows(inp, cfg, np.arange(cfg.rows))
    check_close(y.reshape(cfg.rows, -1), y_ref, True, "after timeout")


# ---------------------------------------------------------------- exact zero-order hold

ZOH_VARIANTS = [("auto", ss.SS_VARIANT_AUTO, 0, 0), ("chained", ss.SS_VARIANT_ROWS, 2, 0),
                ("chunked", ss.SS_VARIANT_CHUNKED, 0, 3), ("seq", ss.SS_VARIANT_ROWS, 1, 0),
                ("simple", ss.SS_VARIANT_SIMPLE, 0, 0)]


@pytest.mark.parametrize("N,L,dt", [(16, 256, "bf16"), (16, 256, "f32"), (16, 100, "f32"),
                                    (4, 64, "f32"), (16, 2048, "bf16")])
@pytest.mark.parametrize("name,variant,tpr,segments", ZOH_VARIANTS, ids=[v[0] for v in ZOH_VARIANTS])
def test_zoh_scan(N, L, dt, name, variant, tpr, segments):
    """SS_DISC_ZOH: the input matrix (exp(dt A) - 1) / A * B, against the
    oracle's ZOH, on every kernel that takes it (the pair-row kernels only
    where their shape rules hold: dstate 16, L a multiple of 16)."""
    pair = name in ("chained", "chunked")
    if pair and (N != 16 or L % 16):
        pytest.skip("the pair-row kernels take dstate 16 and whole 16-step tiles")
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=2, dim=64, dstate=N, seqlen=L,
                           in_dtype=dt, seed=90 + N + L)
    inp = workloads.scan_inputs(cfg, with_h0=True)
    t = device_inputs(inp, cfg)
    ctx = _ctx(variant, tpr, segments)
    ctx.set_option(ss.SS_OPT_DISCRETIZATION, ss.SS_DISC_ZOH)
    y, hl = _run(cfg, t, ctx, h0=t["h0"])
    if pair:
        assert ctx.last_launch()[0] == variant
    rows = np.arange(cfg.rows)
    A = inp["A"]
    y_ref, h_ref = oracle.scan_fwd(inp["u"], inp["delta"], A, inp["B"], inp["C"], D=inp["D"],
                                   delta_bias=inp["delta_bias"], z=inp["z"], h0=inp["h0"],
                                   rows=rows, dim=cfg.dim, zoh=True)
    check_close(y.reshape(cfg.rows, -1), y_ref, dt == "bf16", "y")
    check_close(hl.reshape(cfg.rows, -1), h_ref, dt == "bf16", "h_last")
    # and it is not the simplified result
    y_s, _ = oracle_rows(inp, cfg, rows, h0=inp["h0"])
    assert np.max(np.abs(y_s - y_ref)) > 1e-3 * np.max(np.abs(y_ref))


def test_zoh_small_and_zero_decay_rates():
    """ZOH where dt a is tiny (the series branch of the pair kernels) and
    exactly zero (A = 0: the factor is dt), fp32 inputs against the oracle."""
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=1, dim=64, seqlen=128,
                           in_dtype="f32", seed=97)
    inp = workloads.scan_inputs(cfg, with_h0=True)
    A = inp["A"].copy()
    A[:, 0] = 0.0                    # no decay at all
    A[:, 1] = -1e-4                  # dt a far inside the series range
    A[:, 2] = -0.125 / 0.05          # near the switch for typical dt
    inp["A"] = A
    t = device_inputs(inp, cfg)
    for variant, tpr, seg in ((ss.SS_VARIANT_ROWS, 2, 0), (ss.SS_VARIANT_CHUNKED, 0, 2)):
        ctx = _ctx(variant, tpr, seg)
        ctx.set_option(ss.SS_OPT_DISCRETIZATION, ss.SS_DISC_ZOH)
        y, hl = _run(cfg, t, ctx, h0=t["h0"])
        rows = np.arange(cfg.rows)
        y_ref, h_ref = oracle.scan_fwd(inp["u"], inp["delta"], A, inp["B"], inp["C"], D=inp["D"],
                                       delta_bias=inp["delta_bias"], z=inp["z"], h0=inp["h0"],
                                       rows=rows, dim=cfg.dim, zoh=True)
        check_close(y.reshape(cfg.rows, -1), y_ref, False, "y")
        check_close(hl.reshape(cfg.rows, -1), h_ref, False, "h_last")


def test_zoh_split_row_kernel_unsupported():
    """The 4-thread split-row kernel does not take the zero-order hold."""
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=1, dim=64, seqlen=256, seed=95)
    inp = workloads.scan_inputs(cfg)
    t = device_inputs(inp, cfg)
    ctx = _ctx(ss.SS_VARIANT_ROWS, 4)
    ctx.set_option(ss.SS_OPT_DISCRETIZATION, ss.SS_DISC_ZOH)
    with pytest.raises(ss.SSError) as ei:
        _run(cfg, t, ctx)
    assert ei.value.status == ss.SS_ERR_UNSUPPORTED
