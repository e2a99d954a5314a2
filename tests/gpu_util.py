"""Helpers for the GPU parity tests: move seeded numpy inputs to the device,
run the library, and compare with the fp64 oracle under the stated bounds.

Tolerances (fixed by the problem statement and written here once):
  fp32 inputs:  |y - y_ref| <= 1e-4 * (1 + |y_ref|) elementwise; same for h_last.
  bf16 inputs (fp32 state): max |y - y_ref| <= 1e-2 * max |y_ref| over the
  compared tensor; same for h_last against max |h_ref|.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

F32_RTOL = 1e-4
BF16_REL_MAX = 1e-2


def dev_tensor(a: np.ndarray, device="cuda"):
    """uint16 arrays are bf16 bit patterns; float32 stays float32."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(a).to(device)


def check_close(got, ref, bf16: bool, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite values" % what
    if got.size == 0:
        return 0.0
    if bf16:
        scale = float(np.max(np.abs(ref)))
        err = float(np.max(np.abs(got - ref)))
        assert err <= BF16_REL_MAX * scale + 1e-30, "%s: max err %.3g > %.3g" % (
            what, err, BF16_REL_MAX * scale)
        return err / max(scale, 1e-30)
    excess = np.abs(got - ref) - F32_RTOL * (1.0 + np.abs(ref))
    worst = int(np.argmax(excess))
    assert excess.flat[worst] <= 0, "%s: |%g - %g| at flat %d" % (
        what, got.flat[worst], ref.flat[worst], worst)
    return float(np.max(np.abs(got - ref) / (1.0 + np.abs(ref))))


def device_inputs(inp: dict, cfg, device="cuda"):
    """Full-tensor inputs (rows=None) from workloads.scan_inputs on the device."""
    shp = (cfg.batch, cfg.dim, cfg.seqlen)
    t = {k: dev_tensor(inp[k].reshape(shp), device) for k in ("u", "delta", "z")}
    t["B"] = dev_tensor(inp["B"], device)
    t["C"] = dev_tensor(inp["C"], device)
    for k in ("A", "D", "delta_bias"):
        t[k] = torch.from_numpy(inp[k]).to(device)
    if "h0" in inp:
        t["h0"] = torch.from_numpy(inp["h0"].reshape(cfg.batch, cfg.dim, cfg.dstate)).to(device)
    return t


def oracle_rows(inp: dict, cfg, rows, with_z=True, with_D=True, with_bias=True, h0=None,
                softplus=True):
    """Oracle on selected rows, reading the full-input dict (rows=None draw)."""
    rows = np.asarray(rows)
    u = inp["u"][rows]
    return oracle.scan_fwd(u, inp["delta"][rows], inp["A"], inp["B"], inp["C"],
                           D=inp["D"] if with_D else None,
                           delta_bias=inp["delta_bias"] if with_bias else None,
                           z=inp["z"][rows] if with_z else None, delta_softplus=softplus,
                           h0=None if h0 is None else h0[rows], rows=rows, dim=cfg.dim)


def sample_rows(cfg, n, seed=123):
    g = np.random.default_rng(seed)
    pick = set(g.choice(cfg.rows, size=min(n, cfg.rows), replace=False).tolist())
    pick.update({0, cfg.rows - 1, cfg.dim - 1, min(cfg.dim, cfg.rows - 1)})
    return np.array(sorted(pick))
