"""Seeded synthetic inputs for the selective scan (S6) and its decode update.

This module is the only code shared by the CPU oracle and the CUDA path. It
draws input tensors and nothing else: no discretisation, recurrence, softplus,
contraction or gating happens here.

Shapes follow the problem statement of the selective scan:
  u, delta, z : (batch, dim, seqlen)      dim = d_inner
  B, C        : (batch, dstate, seqlen)   input-dependent, shared over dim
  A           : (dim, dstate) fp32, real and negative
  D, bias     : (dim,) fp32
The workloads mirror the shapes the pages talk about: the 2.8B model block
(d_model 2560, expand 2 -> d_inner 5120, d_state 16) from the soft186.com
article "Mamba选择性状态空间机制" (section "基础模型构建"); million-length
sequences from "Mamba: Linear-Time Sequence Modeling with Selective State
Spaces" (section "Results"); the Mamba-130M block width (d_inner 1536).

Every random stream is keyed by (seed, tensor id, row), so any subset of rows
can be regenerated on its own and is bit-identical to the same rows of a full
draw. bf16 inputs are float32 normal draws rounded to nearest-even bf16; they
are returned as uint16 bit patterns.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

# tensor ids used in the stream keys
_T_U, _T_DELTA, _T_Z, _T_B, _T_C, _T_D, _T_BIAS, _T_H0, _T_STATE = range(9)


@dataclasses.dataclass(frozen=True)
class ScanConfig:
    name: str
    batch: int
    dim: int
    dstate: int
    seqlen: int
    in_dtype: str            # "f32" or "bf16" for u, delta, z, B, C
    seed: int
    dt_lo: float             # log-uniform range of the target time step
    dt_hi: float
    delta_softplus: bool = True
    has_z: bool = True
    has_D: bool = True

    @property
    def rows(self) -> int:
        return self.batch * self.dim

    @property
    def elements(self) -> int:
        """batch * dim * seqlen: the unit of the throughput metric."""
        return self.batch * self.dim * self.seqlen


@dataclasses.dataclass(frozen=True)
class DecodeConfig:
    name: str
    batch: int
    dim: int
    dstate: int
    in_dtype: str
    seed: int
    steps: int
    dt_lo: float
    dt_hi: float
    dt_softplus: bool = True


CONFIGS = {
    # tiny case the oracle finishes instantly; fp32 everywhere
    "tiny": ScanConfig("tiny", 1, 16, 4, 64, "f32", 0, 1e-3, 1e-1),
    # Mamba-130M block: d_inner 1536
    "mamba130m": ScanConfig("mamba130m", 8, 1536, 16, 2048, "bf16", 1, 1e-3, 1e-1),
    # Mamba-2.8B block: d_model 2560 x expand 2 = d_inner 5120, d_state 16
    "mamba2p8b": ScanConfig("mamba2p8b", 8, 5120, 16, 2048, "bf16", 2, 1e-3, 1e-1),
    # million-length scan; small time steps so the state carries far
    "long1m": ScanConfig("long1m", 1, 1536, 16, 1 << 20, "bf16", 3, 1e-4, 1e-2),
}

DECODE = DecodeConfig("decode", 128, 5120, 16, "bf16", 4, 1000, 1e-3, 1e-1)


def _rng(*key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(list(key))))


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bf16 (ties to even); returns uint16 bits.

    Inputs here are finite normal draws, so no NaN handling is needed."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_row(seed: int, tensor: int, row: int, n: int, dtype: str) -> np.ndarray:
    v = _rng(seed, tensor, row).standard_normal(n, dtype=np.float32)
    return f32_to_bf16_bits(v) if dtype == "bf16" else v


def _workers() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _fill_rows(out: np.ndarray, seed: int, tensor: int, rows, n: int, dtype: str) -> None:
    rows = list(rows)

    def work(i_lo_hi):
        lo, hi = i_lo_hi
        for i in range(lo, hi):
            out[i] = _normal_row(seed, tensor, rows[i], n, dtype)

    nw = min(_workers(), max(1, len(rows) // 64))
    step = (len(rows) + nw - 1) // nw
    spans = [(i, min(i + step, len(rows))) for i in range(0, len(rows), step)]
    if len(spans) <= 1:
        for s in spans:
            work(s)
        return
    with ThreadPoolExecutor(nw) as ex:
        list(ex.map(work, spans))


def params(cfg) -> dict:
    """A, D and delta_bias (all fp32).

    A[d, n] = -(n + 1) (real, negative, diagonal state matrix).
    D ~ N(0, 1).
    delta_bias = inverse softplus of t, t log-uniform in [dt_lo, dt_hi]: the
    bias of the step-size projection is set so the time step starts in a
    target range ("details fiction and mamba paper", remark on the Delta
    parameter's bias initialisation)."""
    dim, N = cfg.dim, cfg.dstate
    A = np.tile(-(np.arange(N, dtype=np.float32) + 1.0), (dim, 1)).astype(np.float32)
    D = _rng(cfg.seed, _T_D).standard_normal(dim, dtype=np.float32)
    t = np.exp(_rng(cfg.seed, _T_BIAS).uniform(np.log(cfg.dt_lo), np.log(cfg.dt_hi), dim))
    bias = np.log(np.expm1(t)).astype(np.float32)
    return {"A": np.ascontiguousarray(A), "D": D, "delta_bias": bias}


def scan_inputs(cfg: ScanConfig, rows=None, with_h0: bool = False) -> dict:
    """Draw u, delta, z (per row), B, C (per batch) and the parameters.

    rows: None for every row (row = b * dim + d), else an iterable of row
    indices; u/delta/z then hold only those rows, shape (len(rows), seqlen),
    and B/C still hold every batch.
    Returns numpy arrays; bf16 tensors are uint16 bit patterns."""
    L, N = cfg.seqlen, cfg.dstate
    sel = np.arange(cfg.rows) if rows is None else np.asarray(list(rows), dtype=np.int64)
    dt = np.uint16 if cfg.in_dtype == "bf16" else np.float32
    out = {}
    for name, tid in (("u", _T_U), ("delta", _T_DELTA), ("z", _T_Z)):
        a = np.empty((len(sel), L), dtype=dt)
        _fill_rows(a, cfg.seed, tid, sel.tolist(), L, cfg.in_dtype)
        out[name] = a
    for name, tid in (("B", _T_B), ("C", _T_C)):
        a = np.empty((cfg.batch * N, L), dtype=dt)
        _fill_rows(a, cfg.seed, tid, range(cfg.batch * N), L, cfg.in_dtype)
        out[name] = a.reshape(cfg.batch, N, L)
    out.update(params(cfg))
    out["rows"] = sel
    if with_h0:
        h0 = np.empty((len(sel), N), dtype=np.float32)
        _fill_rows(h0, cfg.seed, _T_H0, sel.tolist(), N, "f32")
        out["h0"] = h0
    return out


def decode_state0(cfg: DecodeConfig) -> np.ndarray:
    """Initial decode state (batch, dim, dstate) fp32 ~ N(0, 1)."""
    return _rng(cfg.seed, _T_STATE).standard_normal(
        (cfg.batch, cfg.dim, cfg.dstate), dtype=np.float32)


def decode_step_inputs(cfg: DecodeConfig, step: int) -> dict:
    """Fresh per-step draws: x, dt, z (batch, dim) and B, C (batch, dstate),
    all ~ N(0, 1) in cfg.in_dtype."""
    out = {}
    for name, tid, shape in (("x", _T_U, (cfg.batch, cfg.dim)),
                             ("dt", _T_DELTA, (cfg.batch, cfg.dim)),
                             ("z", _T_Z, (cfg.batch, cfg.dim)),
                             ("B", _T_B, (cfg.batch, cfg.dstate)),
                             ("C", _T_C, (cfg.batch, cfg.dstate))):
        v = _rng(cfg.seed, 1000 + step, tid).standard_normal(shape, dtype=np.float32)
        out[name] = f32_to_bf16_bits(v) if cfg.in_dtype == "bf16" else v
    return out


def scaled(cfg: ScanConfig, **changes) -> ScanConfig:
    """Same recipe with some fields replaced (e.g. a smaller seqlen)."""
    return dataclasses.replace(cfg, **changes)
