"""Mamba-2 SSD forward on the GPU against the fp64 scan oracle.

SSD computes the selective recurrence with A = a_h for every state of head h,
dt shared by the head's channels and B, C shared by all heads; channel
d = h * headdim + p of the scan oracle is (head h, channel p) of SSD."""
import numpy as np
import pytest
import torch

import oracle
import selective_state_space_136_b300 as ss
from gpu_util import check_close

pytestmark = pytest.mark.gpu


def _bf16(a):
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t, t.view(torch.int16).numpy().view(np.uint16)


def _case(seed, batch, L, H, N, P=64):
    g = np.random.default_rng(seed)
    x, x_bits = _bf16(g.standard_normal((batch, L, H, P)))
    dt_raw, dt_bits = _bf16(g.standard_normal((batch, L, H)) * 0.5 - 1.0)
    B, B_bits = _bf16(g.standard_normal((batch, L, N)) * 0.3)
    C, C_bits = _bf16(g.standard_normal((batch, L, N)) * 0.3)
    A = -g.uniform(0.5, 4.0, H).astype(np.float32)
    D = g.standard_normal(H).astype(np.float32)
    bias = np.log(np.expm1(np.exp(g.uniform(np.log(1e-3), np.log(1e-1), H)))).astype(np.float32)
    h0 = g.standard_normal((batch, H, P, N)).astype(np.float32)
    return dict(x=x, dt=dt_raw, B=B, C=C, A=A, D=D, bias=bias, h0=h0,
                bits=dict(x=x_bits, dt=dt_bits, B=B_bits, C=C_bits))


def _sub(c, b, h):
    """The case restricted to batch b and head h (heads are independent)."""
    bits = c["bits"]
    return dict(x=c["x"][b:b + 1, :, h:h + 1], dt=c["dt"][b:b + 1, :, h:h + 1],
                B=c["B"][b:b + 1], C=c["C"][b:b + 1], A=c["A"][h:h + 1], D=c["D"][h:h + 1],
                bias=c["bias"][h:h + 1], h0=c["h0"][b:b + 1, h:h + 1],
                bits=dict(x=bits["x"][b:b + 1, :, h:h + 1], dt=bits["dt"][b:b + 1, :, h:h + 1],
                          B=bits["B"][b:b + 1], C=bits["C"][b:b + 1]))


def _ctx(path):
    ctx = ss.Context()
    ctx.set_option(ss.SS_OPT_SSD_PATH, path)
    return ctx


def _run(c, ctx, with_h0=True, **kw):
    cu = lambda t: t.cuda()
    y, hl = ss.ss_ssd_fwd(cu(c["x"]), cu(c["dt"]), torch.from_numpy(c["A"]).cuda(), cu(c["B"]),
                          cu(c["C"]), D=torch.from_numpy(c["D"]).cuda(),
                          dt_bias=torch.from_numpy(c["bias"]).cuda(),
                          h0=torch.from_numpy(c["h0"]).cuda() if with_h0 else None, ctx=ctx, **kw)
    torch.cuda.synchronize()
    return y, hl


def _oracle(c, batch, L, H, N, P=64, with_h0=True, softplus=True):
    """The same computation as an ss_scan over d = h*P + p channels."""
    bits = c["bits"]
    u = bits["x"].transpose(0, 2, 3, 1).reshape(batch, H * P, L)          # (b, d, l)
    delta = np.repeat(bits["dt"].transpose(0, 2, 1), P, axis=1)          # (b, d, l)
    A = np.repeat(c["A"], P)[:, None].repeat(N, axis=1).astype(np.float32)
    Bs = np.ascontiguousarray(bits["B"].transpose(0, 2, 1))              # (b, n, l)
    Cs = np.ascontiguousarray(bits["C"].transpose(0, 2, 1))
    h0 = c["h0"].reshape(batch, H * P, N).astype(np.float64) if with_h0 else None
    y, hl = oracle.scan_fwd(np.ascontiguousarray(u), np.ascontiguousarray(delta), A, Bs, Cs,
                            D=np.repeat(c["D"], P), delta_bias=np.repeat(c["bias"], P), z=None,
                            h0=h0, delta_softplus=softplus)
    return (y.reshape(batch, H, P, L).transpose(0, 3, 1, 2), hl.reshape(batch, H, P, N))


@pytest.mark.parametrize("batch,L,H,N", [(2, 128, 3, 64), (1, 256, 2, 128), (2, 64, 1, 128),
                                         (1, 1024, 2, 128), (3, 384, 5, 128)])
@pytest.mark.parametrize("with_h0", [True, False])
@pytest.mark.parametrize("path", ["mma_sync", "tcgen05", "auto"])
def test_ssd_matches_scan_oracle(batch, L, H, N, with_h0, path):
    """Both kernels: the mma.sync one and the tensor-memory one (dstate 128,
    seqlen % 128 == 0; other shapes are refused), and AUTO, which takes the
    tensor-memory kernel where it applies and mma.sync elsewhere."""
    c = _case(200 + L + N + H, batch, L, H, N)
    tc_ok = N == 128 and L % 128 == 0
    ctx = _ctx({"mma_sync": ss.SS_SSD_PATH_MMA_SYNC, "tcgen05": ss.SS_SSD_PATH_TCGEN05,
                "auto": ss.SS_SSD_PATH_AUTO}[path])
    if path == "tcgen05" and not tc_ok:
        with pytest.raises(ss.SSError) as ei:
            _run(c, ctx, with_h0)
        assert ei.value.status == ss.SS_ERR_UNSUPPORTED
        return
    y, hl = _run(c, ctx, with_h0)
    tc = path == "tcgen05" or (path == "auto" and tc_ok)
    assert ctx.last_launch()[0] == (1 if tc else 0)
    y_ref, h_ref = _oracle(c, batch, L, H, N, with_h0=with_h0)
    check_close(y.cpu().numpy(), y_ref, True, "y")
    check_close(hl.cpu().numpy(), h_ref, True, "h_last")


def test_ssd_tensor_memory_bf16_output_and_no_softplus():
    """Tensor-memory kernel with bf16 y, and with dt taken as is (positive)."""
    batch, L, H, N = 2, 256, 3, 128
    c = _case(215, batch, L, H, N)
    ctx = _ctx(ss.SS_SSD_PATH_TCGEN05)
    y, hl = _run(c, ctx, out_dtype=torch.bfloat16)
    assert ctx.last_launch()[0] == 1
    y_ref, h_ref = _oracle(c, batch, L, H, N)
    check_close(y.float().cpu().numpy(), y_ref, True, "y bf16")
    check_close(hl.cpu().numpy(), h_ref, True, "h_last")
    g = np.random.default_rng(216)
    dt, dt_bits = _bf16(np.abs(g.standard_normal((batch, L, H))) * 0.05 + 0.01)
    c2 = dict(c, dt=dt, bias=np.zeros(H, np.float32), bits=dict(c["bits"], dt=dt_bits))
    y, hl = _run(c2, ctx, dt_softplus=False)
    assert ctx.last_launch()[0] == 1
    y_ref, h_ref = _oracle(c2, batch, L, H, N, softplus=False)
    check_close(y.cpu().numpy(), y_ref, True, "y no softplus")
    check_close(hl.cpu().numpy(), h_ref, True, "h_last no softplus")


def test_ssd_full_size_sampled_heads():
    """The Mamba-2 block shape (8, 2048, 80 heads x 64, dstate 128) in one call;
    a few (batch, head) pairs against the oracle (heads are independent)."""
    batch, L, H, N = 8, 2048, 80, 128
    c = _case(217, batch, L, H, N)
    refs = {bh: _oracle(_sub(c, *bh), 1, L, 1, N) for bh in ((0, 0), (3, 41), (7, 79))}
    for path, variant in ((ss.SS_SSD_PATH_MMA_SYNC, 0), (ss.SS_SSD_PATH_TCGEN05, 1),
                          (ss.SS_SSD_PATH_AUTO, 1)):
        ctx = _ctx(path)
        y, hl = _run(c, ctx)
        assert ctx.last_launch()[0] == variant
        for (b, h), (y_ref, h_ref) in refs.items():
            check_close(y[b:b + 1, :, h:h + 1].cpu().numpy(), y_ref, True, "y (%d, %d)" % (b, h))
            check_close(hl[b:b + 1, h:h + 1].cpu().numpy(), h_ref, True, "h_last (%d, %d)" % (b, h))


def test_ssd_bf16_output():
    batch, L, H, N = 1, 128, 2, 64
    c = _case(210, batch, L, H, N)
    y, _ = ss.ss_ssd_fwd(c["x"].cuda(), c["dt"].cuda(), torch.from_numpy(c["A"]).cuda(),
                         c["B"].cuda(), c["C"].cuda(), D=torch.from_numpy(c["D"]).cuda(),
                         dt_bias=torch.from_numpy(c["bias"]).cuda(), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    y_ref, _ = _oracle(c, batch, L, H, N, with_h0=False)
    check_close(y.float().cpu().numpy(), y_ref, True, "y")


def test_ssd_split_equals_whole():
    """Two calls with the state handed over equal one call over the whole sequence."""
    batch, L, H, N = 1, 256, 2, 128
    c = _case(211, batch, L, H, N)
    args = lambda a, b_: dict(D=torch.from_numpy(c["D"]).cuda(),
                              dt_bias=torch.from_numpy(c["bias"]).cuda())
    A = torch.from_numpy(c["A"]).cuda()
    x, dt, B, C = (c[k].cuda() for k in ("x", "dt", "B", "C"))
    y, hl = ss.ss_ssd_fwd(x, dt, A, B, C, **args(0, 0))
    y1, h1 = ss.ss_ssd_fwd(x[:, :128].contiguous(), dt[:, :128].contiguous(), A,
                           B[:, :128].contiguous(), C[:, :128].contiguous(), **args(0, 0))
    y2, h2 = ss.ss_ssd_fwd(x[:, 128:].contiguous(), dt[:, 128:].contiguous(), A,
                           B[:, 128:].contiguous(), C[:, 128:].contiguous(), h0=h1, **args(0, 0))
    torch.cuda.synchronize()
    both = torch.cat([y1, y2], dim=1)
    scale = float(y.abs().max())
    assert float((both - y).abs().max()) <= 1e-4 * scale
    assert float((h2 - hl).abs().max()) <= 1e-4 * float(hl.abs().max())


def test_ssd_unsupported_shapes():
    c = _case(212, 1, 96, 1, 64)  # seqlen not a multiple of 64
    with pytest.raises(ss.SSError) as ei:
        ss.ss_ssd_fwd(c["x"].cuda(), c["dt"].cuda(), torch.from_numpy(c["A"]).cuda(),
                      c["B"].cuda(), c["C"].cuda())
    assert ei.value.status == ss.SS_ERR_UNSUPPORTED
