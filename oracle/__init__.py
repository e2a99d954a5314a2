"""fp64 CPU oracle for the selective scan (S6), its decode update, and the
causal depthwise convolution of the Mamba block with its decode step.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only callers. The CUDA library never imports it and
shares no code with it.

The arithmetic lives in ss_oracle.c (plain C, fp64, sequential in time); this
module compiles it with gcc (no fast-math) and wraps it with ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ss_oracle.c")
_LIB = os.path.join(_HERE, "libss_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ss_oracle.c into libss_oracle.so (gcc -O2, IEEE semantics)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC",
                               "-shared", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P, I, LL, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_double
        lib.ss_oracle_scan.argtypes = [LL, P, P, I, I, LL, I, P, P, P, P, P, P, P, P, I, P, P, P, I,
                                       I]
        lib.ss_oracle_scan.restype = I
        lib.ss_oracle_state_update.argtypes = [LL, P, P, I, I, I, P, P, P, P, P, P, P, P, P, I, P,
                                               I, I]
        lib.ss_oracle_state_update.restype = I
        lib.ss_oracle_scan_bwd.argtypes = [LL, P, P, I, I, LL, I, P, P, P, P, P, P, P, P, I, P, I,
                                           P, P, P, P, P, P, P, P, P, P, P]
        lib.ss_oracle_scan_bwd.restype = I
        lib.ss_oracle_conv1d.argtypes = [LL, P, I, LL, I, P, P, P, P, I, P, P]
        lib.ss_oracle_conv1d.restype = I
        lib.ss_oracle_conv1d_update.argtypes = [LL, P, I, I, P, P, P, I, P, P]
        lib.ss_oracle_conv1d_update.restype = I
        lib.ss_oracle_softplus.argtypes = [D]
        lib.ss_oracle_softplus.restype = D
        lib.ss_oracle_silu.argtypes = [D]
        lib.ss_oracle_silu.restype = D
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _cpu_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return 1
    if a.dtype == np.float32:
        return 0
    raise TypeError("oracle inputs are float32 or bf16 bit patterns (uint16), got %s" % a.dtype)


def softplus(x: float) -> float:
    return _load().ss_oracle_softplus(float(x))


def silu(x: float) -> float:
    return _load().ss_oracle_silu(float(x))


def scan_fwd(u, delta, A, B, C, D=None, delta_bias=None, z=None, delta_softplus=True,
             h0=None, rows=None, dim=None, threads=None, zoh=False):
    """Selective scan forward in fp64.

    Full-tensor form: u, delta, z of shape (batch, dim, L); B, C (batch, N, L).
    Row-subset form: pass rows (flat row indices b*dim+d) and dim; u, delta, z
    are then (len(rows), L) holding just those rows.
    A is (dim, N) float32; D and delta_bias (dim,) float32 or None.
    Inputs are float32, or uint16 bf16 bit patterns (all of one kind).
    h0: None (zero state) or (rows..., N).
    zoh: use the exact zero-order-hold input matrix (exp(dt A) - 1) / A * B
    instead of dt * B.
    Returns (y, h_last) in float64, shaped like u and (rows..., N)."""
    u = np.ascontiguousarray(u)
    full = rows is None
    B = np.ascontiguousarray(B)
    batch, N, L = B.shape
    if full:
        batch_u, dim, L_u = u.shape
        assert batch_u == batch and L_u == L
        rows = np.arange(batch * dim)
    else:
        assert dim is not None
        rows = np.asarray(rows, dtype=np.int64)
    nrows = len(rows)
    code = _dtype_code(u)
    flat = lambda a: None if a is None else np.ascontiguousarray(a).reshape(nrows, L)
    u2, d2, z2 = flat(u), flat(delta), flat(z)
    for a in (d2, z2, B, C):
        if a is not None and _dtype_code(a) != code:
            raise TypeError("mixed input dtypes")
    row_b = (rows // dim).astype(np.int32)
    row_d = (rows % dim).astype(np.int32)
    A = np.ascontiguousarray(A, dtype=np.float32)
    assert A.shape == (dim, N)
    Dp = None if D is None else np.ascontiguousarray(D, dtype=np.float32)
    bp = None if delta_bias is None else np.ascontiguousarray(delta_bias, dtype=np.float32)
    h0p = None if h0 is None else np.ascontiguousarray(h0, dtype=np.float64).reshape(nrows, N)
    y = np.empty((nrows, L), dtype=np.float64)
    hl = np.empty((nrows, N), dtype=np.float64)
    C = np.ascontiguousarray(C)
    rc = _load().ss_oracle_scan(nrows, _ptr(row_b), _ptr(row_d), dim, N, L, code, _ptr(u2),
                                _ptr(d2), _ptr(z2), _ptr(A), _ptr(B), _ptr(C), _ptr(Dp),
                                _ptr(bp), int(bool(delta_softplus)), _ptr(h0p), _ptr(y), _ptr(hl),
                                int(bool(zoh)), threads or _cpu_threads())
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    if full:
        return y.reshape(batch, dim, L), hl.reshape(batch, dim, N)
    return y, hl


def state_update(state, x, dt, A, B, C, D=None, dt_bias=None, z=None, dt_softplus=True,
                 rows=None, dim=None, threads=None, zoh=False):
    """One decode step in fp64. state (batch, dim, N) float64 is updated in
    place; x, dt, z are (batch, dim) (or (len(rows),) with rows/dim given);
    B, C are (batch, N). Returns y (float64) shaped like x."""
    B = np.ascontiguousarray(B)
    batch, N = B.shape
    if rows is None:
        dim = x.shape[1]
        rows = np.arange(batch * dim)
    rows = np.asarray(rows, dtype=np.int64)
    nrows = len(rows)
    assert state.dtype == np.float64 and state.flags.c_contiguous and state.size == nrows * N
    code = _dtype_code(np.asarray(x))
    row_b = (rows // dim).astype(np.int32)
    row_d = (rows % dim).astype(np.int32)
    cont = lambda a: None if a is None else np.ascontiguousarray(a)
    x, dt, z, C = cont(x), cont(dt), cont(z), cont(C)
    A = np.ascontiguousarray(A, dtype=np.float32)
    Dp = None if D is None else np.ascontiguousarray(D, dtype=np.float32)
    bp = None if dt_bias is None else np.ascontiguousarray(dt_bias, dtype=np.float32)
    y = np.empty(nrows, dtype=np.float64)
    rc = _load().ss_oracle_state_update(nrows, _ptr(row_b), _ptr(row_d), dim, N, code,
                                        _ptr(state), _ptr(x), _ptr(dt), _ptr(z), _ptr(A),
                                        _ptr(B), _ptr(C), _ptr(Dp), _ptr(bp),
                                        int(bool(dt_softplus)), _ptr(y), int(bool(zoh)),
                                        threads or 1)
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return y.reshape(np.asarray(x).shape)


def conv1d_fwd(x, weight, bias=None, init_state=None, silu=False, rows=None, dim=None):
    """Causal depthwise convolution in fp64.

    Full-tensor form: x (batch, dim, L). Row-subset form: x (len(rows), L) with
    rows (flat indices b*dim+d) and dim. weight (dim, W) float32, bias (dim,)
    float32 or None; init_state None (zeros) or (rows..., W-1), the W-1 inputs
    before step 0, oldest first. x is float32 or bf16 bit patterns (uint16).
    Returns (out, final_state) in float64: out shaped like x, final_state
    (rows..., W-1), the last W-1 inputs."""
    x = np.ascontiguousarray(x)
    weight = np.ascontiguousarray(weight, dtype=np.float32)
    W = weight.shape[1]
    if rows is None:
        batch, dim, L = x.shape
        rows = np.arange(batch * dim)
        out_shape, st_shape = x.shape, (batch, dim, W - 1)
    else:
        rows = np.asarray(rows, dtype=np.int64)
        L = x.shape[-1]
        out_shape, st_shape = (len(rows), L), (len(rows), W - 1)
    nrows = len(rows)
    row_d = (rows % dim).astype(np.int32)
    bp = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    sp = None if init_state is None else \
        np.ascontiguousarray(init_state, dtype=np.float64).reshape(nrows, W - 1)
    out = np.empty((nrows, L), dtype=np.float64)
    fs = np.empty((nrows, max(W - 1, 1)), dtype=np.float64)
    rc = _load().ss_oracle_conv1d(nrows, _ptr(row_d), W, L, _dtype_code(x), _ptr(x),
                                  _ptr(weight), _ptr(bp), _ptr(sp), int(bool(silu)), _ptr(out),
                                  _ptr(fs))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out.reshape(out_shape), fs[:, :W - 1].reshape(st_shape)


def conv_scan_fwd(x, conv_weight, delta, A, B, C, conv_bias=None, conv_init=None, conv_silu=True,
                  D=None, delta_bias=None, z=None, delta_softplus=True, h0=None, rows=None,
                  dim=None):
    """The Mamba block's convolution followed by the selective scan, in that
    order ("Mamba: Linear-Time Sequence Modeling with Selective State Spaces",
    section "Key terms": the block's 1D convolution feeds the SSM): u =
    conv1d_fwd(x, ...) (silu applied when conv_silu), then scan_fwd on u.

    The convolution's fp64 output is handed to the scan as float32 (the scan
    reads float32 or bf16 inputs); delta, z, B and C are widened to float32,
    which is exact for bf16. Same full-tensor or row-subset forms as scan_fwd.
    Returns (y, h_last, u, conv_final_state), u and the state in float64."""
    u, fs = conv1d_fwd(x, conv_weight, bias=conv_bias, init_state=conv_init, silu=conv_silu,
                       rows=rows, dim=dim)
    wide = lambda a: None if a is None else (
        _bf16_to_f32(a) if np.asarray(a).dtype == np.uint16 else np.asarray(a, dtype=np.float32))
    y, h = scan_fwd(u.astype(np.float32), wide(delta), A, wide(B), wide(C), D=D,
                    delta_bias=delta_bias, z=wide(z), delta_softplus=delta_softplus, h0=h0,
                    rows=rows, dim=dim)
    return y, h, u, fs


def _bf16_to_f32(a):
    a = np.ascontiguousarray(a)
    return (a.astype(np.uint32) << 16).view(np.float32)


def conv1d_update(state, x, weight, bias=None, silu=False, dim=None):
    """One decode step of the convolution in fp64. state (batch, dim, W-1)
    float64 (oldest input first) is updated in place; x is (batch, dim).
    Returns out (float64) shaped like x."""
    x = np.ascontiguousarray(x)
    weight = np.ascontiguousarray(weight, dtype=np.float32)
    W = weight.shape[1]
    dim = x.shape[-1] if dim is None else dim
    nrows = x.size
    assert state.dtype == np.float64 and state.flags.c_contiguous and state.size == nrows * (W - 1)
    rows = np.arange(nrows)
    row_d = (rows % dim).astype(np.int32)
    bp = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    out = np.empty(nrows, dtype=np.float64)
    rc = _load().ss_oracle_conv1d_update(nrows, _ptr(row_d), W, _dtype_code(x), _ptr(x),
                                         _ptr(weight), _ptr(bp), int(bool(silu)), _ptr(state),
                                         _ptr(out))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return out.reshape(x.shape)


def scan_bwd(u, delta, A, B, C, dy, D=None, delta_bias=None, z=None, delta_softplus=True,
             h0=None, dh_last=None, zoh=False, threads=1):
    """Gradients of the selective scan in fp64 (full tensors only).

    Same inputs as scan_fwd plus dy (batch, dim, L) and optional dh_last
    (batch, dim, N). Returns a dict with du, ddelta, dz (None without z), dA,
    dB, dC, dD, ddelta_bias and dh0, all float64.

    threads > 1 splits the rows into that many contiguous groups, each run by
    the same C routine on its own rows with its own buffers for the sums over
    rows (dA, dB, dC, dD, ddelta_bias), which are added afterwards: only the
    order of those fp64 additions changes."""
    u = np.ascontiguousarray(u)
    batch, dim, L = u.shape
    B = np.ascontiguousarray(B)
    C = np.ascontiguousarray(C)
    N = B.shape[1]
    nrows = batch * dim
    rows = np.arange(nrows)
    row_b = (rows // dim).astype(np.int32)
    row_d = (rows % dim).astype(np.int32)
    code = _dtype_code(u)
    cont = lambda a: None if a is None else np.ascontiguousarray(a)
    delta, z = cont(delta), cont(z)
    A = np.ascontiguousarray(A, dtype=np.float32)
    Dp = None if D is None else np.ascontiguousarray(D, dtype=np.float32)
    bp = None if delta_bias is None else np.ascontiguousarray(delta_bias, dtype=np.float32)
    h0p = None if h0 is None else np.ascontiguousarray(h0, dtype=np.float64)
    dyp = np.ascontiguousarray(dy, dtype=np.float64)
    dhp = None if dh_last is None else np.ascontiguousarray(dh_last, dtype=np.float64)
    out = dict(du=np.zeros((batch, dim, L)), ddelta=np.zeros((batch, dim, L)),
               dz=np.zeros((batch, dim, L)) if z is not None else None,
               dA=np.zeros((dim, N)), dB=np.zeros((batch, N, L)), dC=np.zeros((batch, N, L)),
               dD=np.zeros(dim), ddelta_bias=np.zeros(dim), dh0=np.zeros((batch, dim, N)))
    lib = _load()

    def run_rows(lo, hi):
        """Rows [lo, hi): per-row outputs written in place, sums returned."""
        sums = dict(dA=np.zeros((dim, N)), dB=np.zeros((batch, N, L)), dC=np.zeros((batch, N, L)),
                    dD=np.zeros(dim), ddelta_bias=np.zeros(dim))
        sl = lambda a, w: None if a is None else a.reshape(nrows, w)[lo:hi]
        view = lambda a: None if a is None else a.reshape(nrows, L)[lo:hi]
        rc = lib.ss_oracle_scan_bwd(
            hi - lo, _ptr(row_b[lo:hi]), _ptr(row_d[lo:hi]), dim, N, L, code,
            _ptr(view(u)), _ptr(view(delta)), _ptr(view(z)), _ptr(A), _ptr(B), _ptr(C),
            _ptr(Dp), _ptr(bp), int(bool(delta_softplus)), _ptr(sl(h0p, N)), int(bool(zoh)),
            _ptr(view(dyp)), _ptr(sl(dhp, N)), _ptr(view(out["du"])), _ptr(view(out["ddelta"])),
            _ptr(view(out["dz"])), _ptr(sums["dA"]), _ptr(sums["dB"]), _ptr(sums["dC"]),
            _ptr(sums["dD"]), _ptr(sums["ddelta_bias"]), _ptr(sl(out["dh0"], N)))
        if rc != 0:
            raise ValueError("oracle rejected its arguments")
        return sums

    groups = max(1, min(int(threads), nrows))
    bounds = [(nrows * k // groups, nrows * (k + 1) // groups) for k in range(groups)]
    if groups == 1:
        parts = [run_rows(0, nrows)]
    else:
        from concurrent.futures import ThreadPoolExecutor
        with ThreadPoolExecutor(groups) as ex:
            parts = list(ex.map(lambda b: run_rows(*b), bounds))
    for k in ("dA", "dB", "dC", "dD", "ddelta_bias"):
        out[k] = parts[0][k]
        for part in parts[1:]:
            out[k] += part[k]
    return out
