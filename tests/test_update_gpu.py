"""GPU parity of ss_state_update (decode) against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_util import check_close, dev_tensor

pytestmark = pytest.mark.gpu

ss = pytest.importorskip("selective_state_space_136_b300")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _step_tensors(st):
    return {k: dev_tensor(v) for k, v in st.items()}


@pytest.mark.parametrize("N", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_update_small(N, dt):
    cfg = workloads.DecodeConfig("small", 3, 37, N, dt, 60 + N, 5, 1e-3, 1e-1)
    par = workloads.params(cfg)
    state = workloads.decode_state0(cfg)
    st_dev = torch.from_numpy(state).cuda()
    ref_state = state.astype(np.float64).copy()
    A, D, bias = (torch.from_numpy(par[k]).cuda() for k in ("A", "D", "delta_bias"))
    for step in range(cfg.steps):
        s = workloads.decode_step_inputs(cfg, step)
        t = _step_tensors(s)
        with_z = step % 2 == 0
        y = ss.ss_state_update(st_dev, t["x"], t["dt"], A, t["B"], t["C"], D=D, dt_bias=bias,
                               z=t["z"] if with_z else None)
        y_ref = oracle.state_update(ref_state, s["x"], s["dt"], par["A"], s["B"], s["C"],
                                    D=par["D"], dt_bias=par["delta_bias"],
                                    z=s["z"] if with_z else None)
        torch.cuda.synchronize()
        bf = dt == "bf16"
        check_close(y.cpu().numpy(), y_ref, bf, "y step %d" % step)
        check_close(st_dev.cpu().numpy(), ref_state, bf, "state step %d" % step)


def test_update_chain_equals_scan():
    """k chained GPU decode steps agree with the oracle scan of length k."""
    k = 24
    cfg = workloads.scaled(workloads.CONFIGS["mamba130m"], batch=2, dim=48, seqlen=k, seed=61)
    inp = workloads.scan_inputs(cfg, with_h0=True)
    shp = (cfg.batch, cfg.dim, k)
    u, dl, z = (dev_tensor(inp[n].reshape(shp)) for n in ("u", "delta", "z"))
    B, C = dev_tensor(inp["B"]), dev_tensor(inp["C"])
    A, D, bias = (torch.from_numpy(inp[n]).cuda() for n in ("A", "D", "delta_bias"))
    state = torch.from_numpy(inp["h0"].reshape(cfg.batch, cfg.dim, cfg.dstate)).cuda()
    ys = []
    for t in range(k):
        ys.append(ss.ss_state_update(state, u[..., t].contiguous(), dl[..., t].contiguous(), A,
                                     B[..., t].contiguous(), C[..., t].contiguous(), D=D,
                                     dt_bias=bias, z=z[..., t].contiguous()))
    torch.cuda.synchronize()
    y_ref, h_ref = oracle.scan_fwd(inp["u"].reshape(shp), inp["delta"].reshape(shp), inp["A"],
                                   inp["B"], inp["C"], D=inp["D"], delta_bias=inp["delta_bias"],
                                   z=inp["z"].reshape(shp),
                                   h0=inp["h0"].reshape(cfg.batch, cfg.dim, cfg.dstate))
    check_close(torch.stack(ys, -1).cpu().numpy(), y_ref, True, "chain y")
    check_close(state.cpu().numpy(), h_ref, True, "chain state")


def test_decode_config_1000_chained_steps():
    """The decode workload: batch 128, dim 5120, N 16, fp32 state in place,
    1000 steps with fresh bf16 inputs; sampled rows checked at every step and
    the sampled state after the last."""
    cfg = workloads.DECODE
    par = workloads.params(cfg)
    state0 = workloads.decode_state0(cfg)
    st_dev = torch.from_numpy(state0).cuda()
    g = np.random.default_rng(7)
    rows = np.sort(g.choice(cfg.batch * cfg.dim, size=256, replace=False))
    ref_state = state0.reshape(-1, cfg.dstate)[rows].astype(np.float64).copy()
    A, D, bias = (torch.from_numpy(par[k]).cuda() for k in ("A", "D", "delta_bias"))
    rows_t = torch.from_numpy(rows).cuda()
    worst = 0.0
    for step in range(cfg.steps):
        s = workloads.decode_step_inputs(cfg, step)
        t = _step_tensors(s)
        y = ss.ss_state_update(st_dev, t["x"], t["dt"], A, t["B"], t["C"], D=D, dt_bias=bias,
                               z=t["z"])
        flat = lambda a: a.reshape(-1)[rows]
        y_ref = oracle.state_update(ref_state, flat(s["x"]), flat(s["dt"]), par["A"], s["B"],
                                    s["C"], D=par["D"], dt_bias=par["delta_bias"], z=flat(s["z"]),
                                    rows=rows, dim=cfg.dim)
        yv = y.reshape(-1)[rows_t].cpu().numpy()
        worst = max(worst, check_close(yv, y_ref, True, "decode y step %d" % step))
    sv = st_dev.reshape(-1, cfg.dstate)[rows_t].cpu().numpy()
    check_close(sv, ref_state, True, "decode state after %d steps" % cfg.steps)


@pytest.mark.parametrize("N", [4, 16])
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_update_zoh(N, dt):
    """SS_DISC_ZOH decode steps against the oracle's exact zero-order hold."""
    cfg = workloads.DecodeConfig("small", 3, 37, N, dt, 70 + N, 5, 1e-3, 1e-1)
    par = workloads.params(cfg)
    state = workloads.decode_state0(cfg)
    st_dev = torch.from_numpy(state).cuda()
    ref_state = state.astype(np.float64).copy()
    A, D, bias = (torch.from_numpy(par[k]).cuda() for k in ("A", "D", "delta_bias"))
    ctx = ss.Context(0)
    ctx.set_option(ss.SS_OPT_DISCRETIZATION, ss.SS_DISC_ZOH)
    for step in range(cfg.steps):
        s = workloads.decode_step_inputs(cfg, step)
        t = _step_tensors(s)
        y = ss.ss_state_update(st_dev, t["x"], t["dt"], A, t["B"], t["C"], D=D, dt_bias=bias,
                               z=t["z"], ctx=ctx)
        y_ref = oracle.state_update(ref_state, s["x"], s["dt"], par["A"], s["B"], s["C"],
                                    D=par["D"], dt_bias=par["delta_bias"], z=s["z"], zoh=True)
        torch.cuda.synchronize()
        bf = dt == "bf16"
        check_close(y.cpu().numpy(), y_ref, bf, "y step %d" % step)
        check_close(st_dev.cpu().numpy(), ref_state, bf, "state step %d" % step)
