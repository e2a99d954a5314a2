"""The convolution fused in front of the scan (ss_conv_scan_fwd) against the
oracle's composition conv1d -> scan, on every path of the chained pair-row
kernel: one chained pass (including row blocks split between ranges, whose
tail pieces take the convolution's history from x itself), the chunked
variant, the benchmark shape, and the edge cases."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_136_b300 as ss
import workloads
from gpu_util import check_close, device_inputs, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _conv_params(cfg, W, seed, with_bias=True, with_init=True):
    g = np.random.default_rng(seed)
    w = (g.standard_normal((cfg.dim, W)) * 0.5).astype(np.float32)
    b = (g.standard_normal(cfg.dim) * 0.1).astype(np.float32) if with_bias else None
    init = g.standard_normal((cfg.batch, cfg.dim, W - 1)).astype(np.float32) if with_init else None
    return w, b, init


def _ctx(variant, segments=0):
    c = ss.Context(0)
    c.set_option(ss.SS_OPT_VARIANT, variant)
    c.set_option(ss.SS_OPT_THREADS_PER_ROW, 2 if variant == ss.SS_VARIANT_ROWS else 0)
    c.set_option(ss.SS_OPT_SEGMENTS, segments)
    return c


def _fused(cfg, inp, t, w, b, init, silu, ctx, with_h0=False):
    cuda = lambda a: None if a is None else torch.from_numpy(a).cuda()
    outs = ss.ss_conv_scan_fwd(t["u"], cuda(w), t["delta"], t["A"], t["B"], t["C"],
                               conv_bias=cuda(b), conv_init=cuda(init), conv_silu=silu,
                               D=t["D"], delta_bias=t["delta_bias"], z=t["z"],
                               h0=t.get("h0") if with_h0 else None, return_u=True,
                               return_conv_state=True, ctx=ctx)
    torch.cuda.synchronize()
    assert ctx.device_error() == ss.SS_OK
    return [o.float().cpu().numpy().astype(np.float64) for o in outs]


def _reference(cfg, inp, w, b, init, silu, rows=None, with_h0=False):
    shp = (cfg.batch, cfg.dim, cfg.seqlen)
    h0 = inp["h0"].reshape(cfg.batch, cfg.dim, cfg.dstate) if with_h0 else None
    if rows is None:
        return oracle.conv_scan_fwd(inp["u"].reshape(shp), w, inp["delta"].reshape(shp), inp["A"],
                                    inp["B"], inp["C"], conv_bias=b, conv_init=init,
                                    conv_silu=silu, D=inp["D"], delta_bias=inp["delta_bias"],
                                    z=inp["z"].reshape(shp), h0=h0)
    rows = np.asarray(rows)
    init_r = None if init is None else init.reshape(cfg.rows, -1)[rows]
    return oracle.conv_scan_fwd(inp["u"][rows], w, inp["delta"][rows], inp["A"], inp["B"],
                                inp["C"], conv_bias=b, conv_init=init_r, conv_silu=silu,
                                D=inp["D"], delta_bias=inp["delta_bias"], z=inp["z"][rows],
                                rows=rows, dim=cfg.dim)


def _check_all(cfg, got, ref, bf16, rows=None):
    y, h, u, cs = got
    y_r, h_r, u_r, cs_r = ref
    flat = lambda a, w: a.reshape(cfg.rows, w) if rows is None else a.reshape(cfg.rows, w)[rows]
    check_close(flat(y, cfg.seqlen), y_r.reshape(-1, cfg.seqlen), bf16, "y")
    check_close(flat(h, cfg.dstate), h_r.reshape(-1, cfg.dstate), bf16, "h_last")
    # u as handed back is u rounded to the input dtype
    check_close(flat(u, cfg.seqlen), u_r.reshape(-1, cfg.seqlen), True, "u_out")
    # the convolution's final state is the last inputs themselves: exact
    W1 = cs.shape[-1]
    assert np.array_equal(flat(cs, W1), cs_r.reshape(-1, W1)), "conv_state_out"


VARIANTS = [("chained", ss.SS_VARIANT_ROWS, 0), ("chunked", ss.SS_VARIANT_CHUNKED, 3),
            ("auto", ss.SS_VARIANT_AUTO, 0)]


@pytest.mark.parametrize("W", [2, 3, 4])
@pytest.mark.parametrize("silu", [True, False])
@pytest.mark.parametrize("name,variant,segments", VARIANTS, ids=[v[0] for v in VARIANTS])
def test_fused_matches_oracle(W, silu, name, variant, segments):
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=2, dim=64, seqlen=256,
                           seed=300 + W)
    inp = workloads.scan_inputs(cfg)
    t = device_inputs(inp, cfg)
    w, b, init = _conv_params(cfg, W, seed=W)
    got = _fused(cfg, inp, t, w, b, init, silu, _ctx(variant, segments))
    _check_all(cfg, got, _reference(cfg, inp, w, b, init, silu), True)


@pytest.mark.parametrize("with_bias,with_init,with_h0", [(False, False, False), (True, True, True)])
def test_fused_fp32_inputs(with_bias, with_init, with_h0):
    """fp32 inputs: the elementwise bound 1e-4 (1 + |ref|) on y and h_last."""
    cfg = workloads.scaled(workloads.CONFIGS["tiny"], batch=2, dim=40, dstate=16, seqlen=128,
                           seed=311)
    inp = workloads.scan_inputs(cfg, with_h0=True)
    t = device_inputs(inp, cfg)
    w, b, init = _conv_params(cfg, 4, seed=5, with_bias=with_bias, with_init=with_init)
    for variant, seg in ((ss.SS_VARIANT_ROWS, 0), (ss.SS_VARIANT_CHUNKED, 2)):
        got = _fused(cfg, inp, t, w, b, init, True, _ctx(variant, seg), with_h0=with_h0)
        ref = _reference(cfg, inp, w, b, init, True, with_h0=with_h0)
        check_close(got[0].reshape(cfg.rows, -1), ref[0].reshape(cfg.rows, -1), False, "y")
        check_close(got[1].reshape(cfg.rows, -1), ref[1].reshape(cfg.rows, -1), False, "h_last")


def test_fused_split_row_blocks():
    """2048 row blocks for at most 8 chained ranges per SM: row blocks are split
    and their tail pieces start mid-row, reading the convolution's history from
    x; two calls in a row."""
    for seed in (321, 322):
        cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=8, dim=8192, seqlen=64,
                               seed=seed)
        inp = workloads.scan_inputs(cfg)
        t = device_inputs(inp, cfg)
        w, b, init = _conv_params(cfg, 4, seed=seed)
        got = _fused(cfg, inp, t, w, b, init, True, _ctx(ss.SS_VARIANT_ROWS))
        rows = sample_rows(cfg, 64, seed=seed)
        _check_all(cfg, got, _reference(cfg, inp, w, b, init, True, rows=rows), True, rows=rows)


def test_fused_benchmark_shape_sampled():
    """The 2.8B-block shape in the launch configuration the benchmark times."""
    cfg = workloads.CONFIGS["mamba2p8b"]
    inp = workloads.scan_inputs(cfg)
    t = device_inputs(inp, cfg)
    w, b, init = _conv_params(cfg, 4, seed=7)
    got = _fused(cfg, inp, t, w, b, init, True, _ctx(ss.SS_VARIANT_AUTO))
    rows = sample_rows(cfg, 64, seed=8)
    _check_all(cfg, got, _reference(cfg, inp, w, b, init, True, rows=rows), True, rows=rows)


def test_fused_equals_separate_calls():
    """conv1d then scan through the library (u rounded to bf16 in between)
    agrees with the fused call within the bf16 bound."""
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=2, dim=96, seqlen=512, seed=331)
    inp = workloads.scan_inputs(cfg)
    t = device_inputs(inp, cfg)
    w, b, init = _conv_params(cfg, 4, seed=9)
    cuda = lambda a: torch.from_numpy(a).cuda()
    y_f, h_f, _, _ = ss.ss_conv_scan_fwd(t["u"], cuda(w), t["delta"], t["A"], t["B"], t["C"],
                                         conv_bias=cuda(b), conv_init=cuda(init), D=t["D"],
                                         delta_bias=t["delta_bias"], z=t["z"])
    u, _ = ss.ss_conv1d_fwd(t["u"], cuda(w), bias=cuda(b), init_state=cuda(init), silu=True)
    y_s, h_s = ss.ss_scan_fwd(u, t["delta"], t["A"], t["B"], t["C"], D=t["D"],
                              delta_bias=t["delta_bias"], z=t["z"])
    torch.cuda.synchronize()
    check_close(y_f.cpu().numpy(), y_s.cpu().numpy().astype(np.float64), True, "y")
    check_close(h_f.cpu().numpy(), h_s.cpu().numpy().astype(np.float64), True, "h_last")


def test_fused_unsupported_and_empty():
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=1, dim=32, seqlen=24, seed=341)
    inp = workloads.scan_inputs(cfg)
    t = device_inputs(inp, cfg)
    w = torch.ones(cfg.dim, 4, device="cuda")
    with pytest.raises(ss.SSError) as ei:  # seqlen not a multiple of 16
        ss.ss_conv_scan_fwd(t["u"], w, t["delta"], t["A"], t["B"], t["C"])
    assert ei.value.status == ss.SS_ERR_UNSUPPORTED
    with pytest.raises(ss.SSError) as ei:  # width 5
        ss.ss_conv_scan_fwd(t["u"][..., :16].contiguous(), torch.ones(cfg.dim, 5, device="cuda"),
                            t["delta"][..., :16].contiguous(), t["A"],
                            t["B"][..., :16].contiguous(), t["C"][..., :16].contiguous())
    assert ei.value.status == ss.SS_ERR_UNSUPPORTED
    # seqlen 0: h_last = h0 and the convolution's state = its initial state
    e = lambda k, n: torch.empty((cfg.batch, n, 0), dtype=torch.bfloat16, device="cuda")
    h0 = torch.randn(cfg.batch, cfg.dim, cfg.dstate, device="cuda")
    init = torch.randn(cfg.batch, cfg.dim, 3, device="cuda")
    y, hl, _, cs = ss.ss_conv_scan_fwd(e("u", cfg.dim), w, e("d", cfg.dim), t["A"],
                                       e("B", cfg.dstate), e("C", cfg.dstate), conv_init=init,
                                       h0=h0, return_conv_state=True)
    torch.cuda.synchronize()
    assert y.numel() == 0 and torch.equal(hl, h0) and torch.equal(cs, init)
