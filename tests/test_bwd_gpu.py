"""Backward pass on the GPU against the fp64 oracle's gradients."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_136_b300 as ss
import workloads
from gpu_util import BF16_REL_MAX, dev_tensor, device_inputs

pytestmark = pytest.mark.gpu


def _close(got, ref, bf16, what):
    """fp32 inputs: max error within 1e-4 of the largest reference value;
    bf16 inputs: within the bf16 tolerance of it (gradients are sums of many
    terms, so the bound is relative to the tensor's scale)."""
    got = got.detach().cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got)), what
    scale = max(float(np.max(np.abs(ref))), 1e-30)
    err = float(np.max(np.abs(got - ref)))
    tol = (BF16_REL_MAX if bf16 else 1e-4) * scale
    assert err <= tol, "%s: max err %.3g > %.3g (scale %.3g)" % (what, err, tol, scale)


@pytest.mark.parametrize("N,L,dim,dt", [(16, 64, 48, "f32"), (16, 32, 70, "bf16"),
                                        (4, 48, 33, "f32"), (1, 16, 32, "f32"),
                                        (8, 128, 96, "bf16"), (2, 32, 40, "bf16")])
@pytest.mark.parametrize("full", [True, False])
def test_bwd_matches_oracle(N, L, dim, dt, full):
    """Every gradient, with (full) and without the optional inputs."""
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=2, dim=dim, dstate=N, seqlen=L,
                           in_dtype=dt, seed=100 + N + L + dim)
    inp = workloads.scan_inputs(cfg, with_h0=True)
    t = device_inputs(inp, cfg)
    g = np.random.default_rng(7)
    dy = g.standard_normal((cfg.batch, cfg.dim, L))
    dh = g.standard_normal((cfg.batch, cfg.dim, N))
    kw = dict(D=t["D"], delta_bias=t["delta_bias"], z=t["z"], h0=t["h0"],
              dh_last=torch.from_numpy(dh.astype(np.float32)).cuda()) if full else {}
    got = ss.ss_scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"],
                         torch.from_numpy(dy.astype(np.float32)).cuda(), **kw)
    torch.cuda.synchronize()
    okw = dict(D=inp["D"], delta_bias=inp["delta_bias"], z=inp["z"],
               h0=inp["h0"].reshape(cfg.batch, cfg.dim, N),
               dh_last=dh.astype(np.float32).astype(np.float64)) if full else {}
    shp = (cfg.batch, cfg.dim, L)
    ref = oracle.scan_bwd(inp["u"].reshape(shp), inp["delta"].reshape(shp), inp["A"], inp["B"],
                          inp["C"], dy.astype(np.float32).astype(np.float64),
                          **{k: (v.reshape(shp) if k == "z" else v) for k, v in okw.items()})
    bf = dt == "bf16"
    for k in ("du", "ddelta", "dA", "dB", "dC") + (("dz", "dD", "ddelta_bias", "dh0") if full else ()):
        _close(got[k], ref[k], bf, k)
    if not full:
        assert got["dz"] is None and got["dD"] is None and got["dh0"] is None


@pytest.mark.parametrize("N", [16, 1])
def test_bwd_without_softplus(N):
    """dt = delta + bias taken as is: ddelta is then the dt gradient itself."""
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=2, dim=40, dstate=N, seqlen=48,
                           in_dtype="f32", seed=140 + N)
    inp = workloads.scan_inputs(cfg, with_h0=True)
    # keep dt = delta + bias positive and moderate when used as is
    inp["delta"] = (np.abs(inp["delta"]) * 0.05).astype(np.float32)
    inp["delta_bias"] = np.full_like(inp["delta_bias"], 0.01)
    t = device_inputs(inp, cfg)
    g = np.random.default_rng(8)
    dy = g.standard_normal((cfg.batch, cfg.dim, cfg.seqlen))
    got = ss.ss_scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"],
                         torch.from_numpy(dy.astype(np.float32)).cuda(), D=t["D"],
                         delta_bias=t["delta_bias"], z=t["z"], delta_softplus=False)
    torch.cuda.synchronize()
    shp = (cfg.batch, cfg.dim, cfg.seqlen)
    ref = oracle.scan_bwd(inp["u"].reshape(shp), inp["delta"].reshape(shp), inp["A"], inp["B"],
                          inp["C"], dy.astype(np.float32).astype(np.float64), D=inp["D"],
                          delta_bias=inp["delta_bias"], z=inp["z"].reshape(shp),
                          delta_softplus=False)
    for k in ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias"):
        _close(got[k], ref[k], False, k)


def test_bwd_long_rows():
    """256 channels of the 2.8B-block shape at full length L = 2048, bf16:
    128 tiles of checkpoints per row, every gradient against the oracle."""
    cfg = workloads.CONFIGS["mamba2p8b"]
    inp = workloads.scan_inputs(workloads.scaled(cfg, batch=1, dim=256))
    c2 = workloads.scaled(cfg, batch=1, dim=256)
    t = device_inputs(inp, c2)
    dy = torch.randn(1, 256, cfg.seqlen, device="cuda")
    got = ss.ss_scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], dy, D=t["D"],
                         delta_bias=t["delta_bias"], z=t["z"])
    torch.cuda.synchronize()
    ref = oracle.scan_bwd(inp["u"].reshape(1, 256, -1), inp["delta"].reshape(1, 256, -1),
                          inp["A"], inp["B"], inp["C"], dy.cpu().numpy().astype(np.float64),
                          D=inp["D"], delta_bias=inp["delta_bias"],
                          z=inp["z"].reshape(1, 256, -1))
    for k in ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias"):
        _close(got[k], ref[k], True, k)


@pytest.mark.parametrize("zoh", [False, True], ids=["simplified", "zoh"])
def test_bwd_full_shape(zoh):
    """The 2.8B-block shape (8, 5120, 16, 2048), bf16, every gradient: 1280 row
    blocks in one wave and the per-step atomic sums of dB and dC over all 5120
    channels of a batch, against the oracle run on every row (rows split over
    the host's cores, partial sums added); both discretizations."""
    cfg = workloads.CONFIGS["mamba2p8b"]
    inp = workloads.scan_inputs(cfg)
    t = device_inputs(inp, cfg)
    shp = (cfg.batch, cfg.dim, cfg.seqlen)
    dy = np.random.default_rng(11).standard_normal(shp).astype(np.float32)
    ctx = ss.Context(0)
    ctx.set_option(ss.SS_OPT_DISCRETIZATION, ss.SS_DISC_ZOH if zoh else ss.SS_DISC_SIMPLIFIED)
    got = ss.ss_scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], torch.from_numpy(dy).cuda(),
                         D=t["D"], delta_bias=t["delta_bias"], z=t["z"], ctx=ctx)
    torch.cuda.synchronize()
    ref = oracle.scan_bwd(inp["u"].reshape(shp), inp["delta"].reshape(shp), inp["A"], inp["B"],
                          inp["C"], dy.astype(np.float64), D=inp["D"],
                          delta_bias=inp["delta_bias"], z=inp["z"].reshape(shp), zoh=zoh,
                          threads=oracle._cpu_threads())
    for k in ("du", "ddelta", "dz", "dA", "dB", "dC", "dD", "ddelta_bias"):
        _close(got[k], ref[k], True, k)


@pytest.mark.parametrize("N,L,dim,dt", [(16, 64, 48, "f32"), (16, 32, 70, "bf16"),
                                        (4, 48, 33, "f32"), (1, 16, 32, "bf16")])
@pytest.mark.parametrize("full", [True, False])
def test_bwd_zoh_matches_oracle(N, L, dim, dt, full):
    """SS_DISC_ZOH: every gradient of the scan whose input matrix is
    (exp(dt A) - 1) / A * B, against the oracle's ZOH gradients; with full
    inputs state 0 of every channel has A = 0 (the factor's limit dt and its
    A-derivative's limit dt^2 / 2)."""
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=2, dim=dim, dstate=N, seqlen=L,
                           in_dtype=dt, seed=150 + N + L + dim)
    inp = workloads.scan_inputs(cfg, with_h0=True)
    if full:
        inp["A"][:, 0] = 0.0
    t = device_inputs(inp, cfg)
    g = np.random.default_rng(9)
    dy = g.standard_normal((cfg.batch, cfg.dim, L))
    dh = g.standard_normal((cfg.batch, cfg.dim, N))
    ctx = ss.Context(0)
    ctx.set_option(ss.SS_OPT_DISCRETIZATION, ss.SS_DISC_ZOH)
    kw = dict(D=t["D"], delta_bias=t["delta_bias"], z=t["z"], h0=t["h0"],
              dh_last=torch.from_numpy(dh.astype(np.float32)).cuda()) if full else {}
    got = ss.ss_scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"],
                         torch.from_numpy(dy.astype(np.float32)).cuda(), ctx=ctx, **kw)
    torch.cuda.synchronize()
    shp = (cfg.batch, cfg.dim, L)
    okw = dict(D=inp["D"], delta_bias=inp["delta_bias"], z=inp["z"].reshape(shp),
               h0=inp["h0"].reshape(cfg.batch, cfg.dim, N),
               dh_last=dh.astype(np.float32).astype(np.float64)) if full else {}
    args = (inp["u"].reshape(shp), inp["delta"].reshape(shp), inp["A"], inp["B"], inp["C"],
            dy.astype(np.float32).astype(np.float64))
    ref = oracle.scan_bwd(*args, zoh=True, **okw)
    bf = dt == "bf16"
    for k in ("du", "ddelta", "dA", "dB", "dC") + (("dz", "dD", "ddelta_bias", "dh0") if full else ()):
        _close(got[k], ref[k], bf, k)
    # and it is not the simplified backward
    simp = oracle.scan_bwd(*args, **okw)
    assert np.max(np.abs(simp["dA"] - ref["dA"])) > 1e-3 * np.max(np.abs(ref["dA"]))


def test_bwd_host_checks():
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=1, dim=32, seqlen=24, seed=1)
    inp = workloads.scan_inputs(cfg)
    t = device_inputs(inp, cfg)
    dy = torch.zeros(1, 32, 24, device="cuda")
    with pytest.raises(ss.SSError) as ei:  # seqlen not a multiple of 16
        ss.ss_scan_bwd(t["u"], t["delta"], t["A"], t["B"], t["C"], dy)
    assert ei.value.status == ss.SS_ERR_UNSUPPORTED
