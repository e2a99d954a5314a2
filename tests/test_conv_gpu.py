"""Causal depthwise conv1d and its decode step on the GPU against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_136_b300 as ss
from gpu_util import check_close, dev_tensor

pytestmark = pytest.mark.gpu


def _case(seed, batch, dim, L, W, dt, with_state, with_bias=True):
    g = np.random.default_rng(seed)
    x = g.standard_normal((batch, dim, L)).astype(np.float32)
    if dt == "bf16":
        x = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    c = dict(x=x, weight=g.standard_normal((dim, W)).astype(np.float32),
             bias=g.standard_normal(dim).astype(np.float32) if with_bias else None,
             init_state=g.standard_normal((batch, dim, W - 1)).astype(np.float32)
             if with_state else None)
    return c


def _gpu(c, silu, out_dtype=None):
    t = lambda a: None if a is None else dev_tensor(a)
    out, fs = ss.ss_conv1d_fwd(t(c["x"]), t(c["weight"]), bias=t(c["bias"]),
                               init_state=t(c["init_state"]), silu=silu, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), fs.cpu().numpy().astype(np.float64)


def _ref(c, silu):
    st = None if c["init_state"] is None else c["init_state"].astype(np.float64)
    return oracle.conv1d_fwd(c["x"], c["weight"], bias=c["bias"], init_state=st, silu=silu)


@pytest.mark.parametrize("W", [2, 3, 4])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
@pytest.mark.parametrize("L", [64, 37, 8, 2, 1])
@pytest.mark.parametrize("with_state", [False, True])
def test_conv1d_matches_oracle(W, dt, L, with_state):
    """Whole 8-step chunks (L % 8 == 0) and the per-element path (any L), rows
    shorter than the state, widths 2-4, with and without an initial state."""
    c = _case(70 + W + L, 2, 48, L, W, dt, with_state)
    for silu in (False, True):
        out, fs = _gpu(c, silu, out_dtype=torch.float32)
        o_ref, f_ref = _ref(c, silu)
        check_close(out, o_ref, dt == "bf16", "out")
        # the final state is a copy of inputs: exact
        assert np.array_equal(fs, f_ref)


def test_conv1d_bf16_output_and_no_bias():
    c = _case(81, 3, 40, 96, 4, "bf16", True, with_bias=False)
    out, fs = _gpu(c, True, out_dtype=torch.bfloat16)
    o_ref, f_ref = _ref(c, True)
    check_close(out, o_ref, True, "out")
    assert np.array_equal(fs, f_ref)


def test_conv1d_zero_length():
    c = _case(82, 2, 16, 0, 4, "f32", True)
    x = torch.empty((2, 16, 0), device="cuda")
    fs = torch.full((2, 16, 3), float("nan"), device="cuda")
    ss.ss_conv1d_fwd(x, dev_tensor(c["weight"]), init_state=dev_tensor(c["init_state"]),
                     final_state=fs)
    torch.cuda.synchronize()
    assert np.array_equal(fs.cpu().numpy(), c["init_state"])


def test_conv1d_split_with_state():
    """Two calls with the state handed over equal one call."""
    c = _case(83, 2, 64, 80, 4, "bf16", True)
    out, fs = _gpu(c, True)
    x = dev_tensor(c["x"])
    w, b, s0 = dev_tensor(c["weight"]), dev_tensor(c["bias"]), dev_tensor(c["init_state"])
    o1, s1 = ss.ss_conv1d_fwd(x[..., :24].contiguous(), w, bias=b, init_state=s0, silu=True)
    o2, s2 = ss.ss_conv1d_fwd(x[..., 24:].contiguous(), w, bias=b, init_state=s1, silu=True)
    torch.cuda.synchronize()
    both = torch.cat([o1, o2], dim=-1).float().cpu().numpy().astype(np.float64)
    assert np.array_equal(both, out)
    assert np.array_equal(s2.cpu().numpy().astype(np.float64), fs)


@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_conv1d_update_chain(dt):
    """L decode steps equal the forward pass, on the GPU and against the oracle."""
    W, L = 4, 12
    c = _case(84, 3, 80, L, W, dt, True)
    out_fwd, fs_fwd = _gpu(c, True, out_dtype=torch.float32)
    st = dev_tensor(c["init_state"]).clone()
    w, b = dev_tensor(c["weight"]), dev_tensor(c["bias"])
    x = dev_tensor(c["x"])
    steps = []
    ref_state = c["init_state"].astype(np.float64).copy()
    for l in range(L):
        xl = x[..., l].contiguous()
        o = ss.ss_conv1d_update(st, xl, w, bias=b, silu=True, out_dtype=torch.float32)
        steps.append(o)
        ref = oracle.conv1d_update(ref_state, np.ascontiguousarray(c["x"][..., l]), c["weight"],
                                   bias=c["bias"], silu=True)
        torch.cuda.synchronize()
        check_close(o.cpu().numpy().astype(np.float64), ref, dt == "bf16", "step %d" % l)
    torch.cuda.synchronize()
    chain = torch.stack(steps, dim=-1).cpu().numpy().astype(np.float64)
    assert np.allclose(chain, out_fwd, rtol=1e-6, atol=1e-6)
    assert np.array_equal(st.cpu().numpy().astype(np.float64), fs_fwd)
    assert np.array_equal(st.cpu().numpy().astype(np.float64), ref_state)


def test_conv1d_full_size_sampled():
    """The 2.8B-block shape (8, 5120, 2048) in bf16: sampled rows against the oracle."""
    import workloads
    cfg = workloads.CONFIGS["mamba2p8b"]
    g = np.random.default_rng(85)
    x = torch.randn(cfg.batch, cfg.dim, cfg.seqlen, device="cuda").to(torch.bfloat16)
    w = torch.from_numpy(g.standard_normal((cfg.dim, 4)).astype(np.float32)).cuda()
    b = torch.from_numpy(g.standard_normal(cfg.dim).astype(np.float32)).cuda()
    out, fs = ss.ss_conv1d_fwd(x, w, bias=b, silu=True)
    torch.cuda.synchronize()
    rows = np.sort(g.choice(cfg.rows, 64, replace=False))
    xr = x.view(torch.int16).reshape(cfg.rows, cfg.seqlen)[torch.from_numpy(rows).cuda()]
    xr = xr.cpu().numpy().view(np.uint16)
    o_ref, f_ref = oracle.conv1d_fwd(xr, w.cpu().numpy(), bias=b.cpu().numpy(), silu=True,
                                     rows=rows, dim=cfg.dim)
    got = out.reshape(cfg.rows, cfg.seqlen)[torch.from_numpy(rows).cuda()].float().cpu().numpy()
    check_close(got.astype(np.float64), o_ref, True, "out")
    got_fs = fs.reshape(cfg.rows, 3)[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert np.array_equal(got_fs.astype(np.float64), f_ref)


def test_conv1d_host_checks():
    x = torch.zeros(1, 8, 16, device="cuda")
    with pytest.raises(ss.SSError) as ei:
        ss.ss_conv1d_fwd(x, torch.zeros(8, 5, device="cuda"))
    assert ei.value.status == ss.SS_ERR_UNSUPPORTED
    with pytest.raises(ss.SSError) as ei:
        ss.ss_conv1d_fwd(x, torch.zeros(8, 4, device="cuda"), out=x)  # out overlaps x
    assert ei.value.status == ss.SS_ERR_INVALID_ARG
    st = torch.zeros(1, 8, 3, device="cuda")
    with pytest.raises(ss.SSError) as ei:
        ss.ss_conv1d_fwd(x, torch.zeros(8, 4, device="cuda"), init_state=st, final_state=st)
    assert ei.value.status == ss.SS_ERR_INVALID_ARG
