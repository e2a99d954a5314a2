"""Non-finite inputs on the GPU: where the fp64 oracle's outputs are NaN or
infinite, the kernels' are too, and everywhere else they agree within the
usual tolerance.

The pages do not address NaN or Inf; the reading taken is that they propagate
through the recurrence as the arithmetic defines (a NaN input at step l makes
that row's state and every output from step l on NaN; a NaN in B or C reaches
every row of its batch; delta = -inf gives dt = 0, a step that changes
nothing). The oracle side of this is pinned on the CPU in
test_oracle_nonfinite.py.
"""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_136_b300 as ss
import workloads
from gpu_util import BF16_REL_MAX, dev_tensor, device_inputs, oracle_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _bf16(v):
    return workloads.f32_to_bf16_bits(np.array([v], dtype=np.float32))[0]


def _poisoned(cfg, case):
    """Inputs of cfg with one non-finite value planted (bf16 bit patterns)."""
    inp = workloads.scan_inputs(cfg)
    L = cfg.seqlen
    if case == "nan_u":
        inp["u"][1 * cfg.dim + 5, 100] = _bf16(np.nan)
    elif case == "inf_delta":
        inp["delta"][0 * cfg.dim + 9, 37] = _bf16(np.inf)
    elif case == "neg_inf_delta":
        inp["delta"][0 * cfg.dim + 2, 10] = _bf16(-np.inf)
    elif case == "nan_B":
        inp["B"][1, 3, 200 % L] = _bf16(np.nan)
    elif case == "nan_C":
        inp["C"][0, 7, 150 % L] = _bf16(np.nan)
    else:
        raise ValueError(case)
    return inp


def _compare(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    fin_ref = np.isfinite(ref)
    fin_got = np.isfinite(got)
    bad = np.argwhere(fin_ref != fin_got)
    assert bad.size == 0, "%s: finiteness differs at %s (got %s, ref %s)" % (
        what, bad[0], got[tuple(bad[0])], ref[tuple(bad[0])])
    if fin_ref.any():
        scale = float(np.max(np.abs(ref[fin_ref])))
        err = float(np.max(np.abs(got[fin_ref] - ref[fin_ref])))
        assert err <= BF16_REL_MAX * scale, "%s: max err %.3g" % (what, err)
    return int((~fin_ref).sum())


VARIANTS = [("auto", ss.SS_VARIANT_AUTO, 0, 0), ("chained", ss.SS_VARIANT_ROWS, 2, 0),
            ("chunked", ss.SS_VARIANT_CHUNKED, 0, 3), ("seq", ss.SS_VARIANT_ROWS, 1, 0),
            ("rows4", ss.SS_VARIANT_ROWS, 4, 0), ("simple", ss.SS_VARIANT_SIMPLE, 0, 0)]


@pytest.mark.parametrize("case", ["nan_u", "inf_delta", "neg_inf_delta", "nan_B", "nan_C"])
@pytest.mark.parametrize("name,variant,tpr,segments", VARIANTS, ids=[v[0] for v in VARIANTS])
def test_scan_nonfinite_matches_oracle(case, name, variant, tpr, segments):
    cfg = workloads.scaled(workloads.CONFIGS["mamba2p8b"], batch=2, dim=64, seqlen=256, seed=91)
    inp = _poisoned(cfg, case)
    t = device_inputs(inp, cfg)
    ctx = ss.Context(0)
    ctx.set_option(ss.SS_OPT_VARIANT, variant)
    ctx.set_option(ss.SS_OPT_THREADS_PER_ROW, tpr)
    ctx.set_option(ss.SS_OPT_SEGMENTS, segments)
    y, hl = ss.ss_scan_fwd(t["u"], t["delta"], t["A"], t["B"], t["C"], D=t["D"],
                           delta_bias=t["delta_bias"], z=t["z"], ctx=ctx)
    torch.cuda.synchronize()
    assert ctx.device_error() == ss.SS_OK
    rows = np.arange(cfg.rows)
    y_ref, h_ref = oracle_rows(inp, cfg, rows)
    n_bad = _compare(y.cpu().numpy().reshape(cfg.rows, cfg.seqlen), y_ref, "y")
    _compare(hl.cpu().numpy().reshape(cfg.rows, cfg.dstate), h_ref, "h_last")
    if case == "neg_inf_delta":
        assert n_bad == 0  # dt = 0: a step that changes nothing
    else:
        assert n_bad > 0


@pytest.mark.parametrize("what", ["x", "dt", "B", "state"])
def test_decode_nonfinite_matches_oracle(what):
    cfg = workloads.DecodeConfig("nan", 2, 96, 16, "bf16", 17, 1, 1e-3, 1e-1)
    par = workloads.params(cfg)
    s = workloads.decode_step_inputs(cfg, 0)
    st0 = workloads.decode_state0(cfg)
    if what == "x":
        s["x"][1, 7] = _bf16(np.nan)
    elif what == "dt":
        s["dt"][0, 3] = _bf16(np.inf)
    elif what == "B":
        s["B"][1, 5] = _bf16(np.nan)
    else:
        st0[0, 11, 2] = np.nan
    state = torch.from_numpy(st0.copy()).cuda()
    y = ss.ss_state_update(state, dev_tensor(s["x"]), dev_tensor(s["dt"]),
                           torch.from_numpy(par["A"]).cuda(), dev_tensor(s["B"]),
                           dev_tensor(s["C"]), D=torch.from_numpy(par["D"]).cuda(),
                           dt_bias=torch.from_numpy(par["delta_bias"]).cuda(),
                           z=dev_tensor(s["z"]))
    torch.cuda.synchronize()
    ref_state = st0.astype(np.float64)
    y_ref = oracle.state_update(ref_state, s["x"], s["dt"], par["A"], s["B"], s["C"], D=par["D"],
                                dt_bias=par["delta_bias"], z=s["z"])
    assert _compare(y.cpu().numpy(), y_ref, "y") > 0
    _compare(state.cpu().numpy(), ref_state, "state")
