"""Python binding of the ss_scan CUDA library (selective scan S6, sm_103a).

Argument marshalling only: every step of the scan and of the decode update
runs in the CUDA kernels of libss_scan.so, reached through its C ABI
(include/ss_scan.h). PyTorch supplies device memory and the current stream.
There is no CPU fallback: if the library is missing, every call raises.

    from selective_state_space_136_b300 import ss_scan_fwd, ss_state_update
    y, h_last = ss_scan_fwd(u, delta, A, B, C, D=D, delta_bias=bias, z=z)
    y = ss_state_update(state, x, dt, A, B, C, D=D, dt_bias=bias, z=z)
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("SS_SCAN_LIB") or os.path.join(_HERE, "libss_scan.so")

SS_F32, SS_BF16 = 0, 1
SS_OK, SS_ERR_INVALID_ARG, SS_ERR_UNSUPPORTED, SS_ERR_CUDA, SS_ERR_TIMEOUT, SS_ERR_DEVICE = range(6)
SS_VARIANT_AUTO, SS_VARIANT_ROWS, SS_VARIANT_CHUNKED, SS_VARIANT_SIMPLE = range(4)
(SS_OPT_VARIANT, SS_OPT_SEGMENTS, SS_OPT_THREADS_PER_ROW, SS_OPT_WAIT_LIMIT,
 SS_OPT_TEST_DROP_TILE, SS_OPT_RESIDENT_WARPS, SS_OPT_DISCRETIZATION, SS_OPT_SSD_PATH) = range(8)
SS_DISC_SIMPLIFIED, SS_DISC_ZOH = range(2)
SS_SSD_PATH_AUTO, SS_SSD_PATH_MMA_SYNC, SS_SSD_PATH_TCGEN05 = range(3)

_vp = ctypes.c_void_p


class ScanArgs(ctypes.Structure):
    """Mirror of ss_scan_args."""
    _fields_ = [("batch", ctypes.c_int), ("dim", ctypes.c_int), ("dstate", ctypes.c_int),
                ("seqlen", ctypes.c_longlong), ("in_dtype", ctypes.c_int),
                ("out_dtype", ctypes.c_int), ("u", _vp), ("delta", _vp), ("z", _vp),
                ("A", _vp), ("B", _vp), ("C", _vp), ("D", _vp), ("delta_bias", _vp),
                ("delta_softplus", ctypes.c_int), ("h0", _vp), ("y", _vp), ("h_last", _vp)]


class ConvScanArgs(ctypes.Structure):
    """Mirror of ss_conv_scan_args."""
    _fields_ = [("scan", ScanArgs), ("conv_width", ctypes.c_int), ("conv_weight", _vp),
                ("conv_bias", _vp), ("conv_init", _vp), ("conv_silu", ctypes.c_int),
                ("u_out", _vp), ("conv_state_out", _vp)]


class UpdateArgs(ctypes.Structure):
    """Mirror of ss_update_args."""
    _fields_ = [("batch", ctypes.c_int), ("dim", ctypes.c_int), ("dstate", ctypes.c_int),
                ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int), ("state", _vp),
                ("x", _vp), ("dt", _vp), ("z", _vp), ("A", _vp), ("B", _vp), ("C", _vp),
                ("D", _vp), ("dt_bias", _vp), ("dt_softplus", ctypes.c_int), ("y", _vp)]


class ScanBwdArgs(ctypes.Structure):
    """Mirror of ss_scan_bwd_args."""
    _fields_ = [("batch", ctypes.c_int), ("dim", ctypes.c_int), ("dstate", ctypes.c_int),
                ("seqlen", ctypes.c_longlong), ("in_dtype", ctypes.c_int), ("u", _vp),
                ("delta", _vp), ("z", _vp), ("A", _vp), ("B", _vp), ("C", _vp), ("D", _vp),
                ("delta_bias", _vp), ("delta_softplus", ctypes.c_int), ("h0", _vp), ("dy", _vp),
                ("dh_last", _vp), ("du", _vp), ("ddelta", _vp), ("dz", _vp), ("dA", _vp),
                ("dB", _vp), ("dC", _vp), ("dD", _vp), ("ddelta_bias", _vp), ("dh0", _vp)]


class SsdArgs(ctypes.Structure):
    """Mirror of ss_ssd_args."""
    _fields_ = [("batch", ctypes.c_int), ("heads", ctypes.c_int), ("headdim", ctypes.c_int),
                ("dstate", ctypes.c_int), ("seqlen", ctypes.c_longlong),
                ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int), ("x", _vp),
                ("dt", _vp), ("A", _vp), ("B", _vp), ("C", _vp), ("D", _vp), ("dt_bias", _vp),
                ("dt_softplus", ctypes.c_int), ("h0", _vp), ("y", _vp), ("h_last", _vp)]


class Conv1dArgs(ctypes.Structure):
    """Mirror of ss_conv1d_args."""
    _fields_ = [("batch", ctypes.c_int), ("dim", ctypes.c_int), ("width", ctypes.c_int),
                ("seqlen", ctypes.c_longlong), ("in_dtype", ctypes.c_int),
                ("out_dtype", ctypes.c_int), ("x", _vp), ("weight", _vp), ("bias", _vp),
                ("init_state", _vp), ("silu", ctypes.c_int), ("out", _vp),
                ("final_state", _vp)]


class Conv1dUpdateArgs(ctypes.Structure):
    """Mirror of ss_conv1d_update_args."""
    _fields_ = [("batch", ctypes.c_int), ("dim", ctypes.c_int), ("width", ctypes.c_int),
                ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int), ("state", _vp),
                ("x", _vp), ("weight", _vp), ("bias", _vp), ("silu", ctypes.c_int),
                ("out", _vp)]


class SSError(RuntimeError):
    def __init__(self, status, what):
        super().__init__("%s: %s (status %d)" % (what, status_string(status), status))
        self.status = status


_lib = None
_lib_lock = threading.Lock()


def lib():
    """The loaded libss_scan.so (raises if it has not been built)."""
    global _lib
    with _lib_lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError("libss_scan.so is missing: build it with "
                                   "`python -m selective_state_space_136_b300.build`")
            L = ctypes.CDLL(LIB_PATH)
            L.ss_create.argtypes = [ctypes.POINTER(_vp), ctypes.c_int]
            L.ss_destroy.argtypes = [_vp]
            L.ss_scan_fwd.argtypes = [_vp, ctypes.POINTER(ScanArgs), _vp]
            L.ss_conv_scan_fwd.argtypes = [_vp, ctypes.POINTER(ConvScanArgs), _vp]
            L.ss_state_update.argtypes = [_vp, ctypes.POINTER(UpdateArgs), _vp]
            L.ss_conv1d_fwd.argtypes = [_vp, ctypes.POINTER(Conv1dArgs), _vp]
            L.ss_scan_bwd.argtypes = [_vp, ctypes.POINTER(ScanBwdArgs), _vp]
            L.ss_ssd_fwd.argtypes = [_vp, ctypes.POINTER(SsdArgs), _vp]
            L.ss_conv1d_update.argtypes = [_vp, ctypes.POINTER(Conv1dUpdateArgs), _vp]
            L.ss_get_device_error.argtypes = [_vp, _vp]
            L.ss_status_string.argtypes = [ctypes.c_int]
            L.ss_status_string.restype = ctypes.c_char_p
            L.ss_set_option.argtypes = [_vp, ctypes.c_int, ctypes.c_longlong]
            L.ss_last_launch.argtypes = [_vp, ctypes.POINTER(ctypes.c_int),
                                         ctypes.POINTER(ctypes.c_int)]
            for f in ("ss_create", "ss_destroy", "ss_scan_fwd", "ss_conv_scan_fwd", "ss_state_update",
                      "ss_get_device_error", "ss_set_option", "ss_last_launch"):
                getattr(L, f).restype = ctypes.c_int
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().ss_status_string(int(status)).decode()


def _check(rc, what):
    if rc != SS_OK:
        raise SSError(rc, what)


class Context:
    """Owns one ss_ctx (bound to one device)."""

    def __init__(self, device: int = 0):
        self._h = _vp()
        _check(lib().ss_create(ctypes.byref(self._h), int(device)), "ss_create")
        self.device = int(device)

    @property
    def handle(self):
        return self._h

    def set_option(self, option: int, value: int):
        _check(lib().ss_set_option(self._h, int(option), int(value)), "ss_set_option")

    def device_error(self, stream=None) -> int:
        return lib().ss_get_device_error(self._h, _stream_ptr(stream, self.device))

    def last_launch(self):
        v, n = ctypes.c_int(), ctypes.c_int()
        _check(lib().ss_last_launch(self._h, ctypes.byref(v), ctypes.byref(n)), "ss_last_launch")
        return v.value, n.value

    def close(self):
        if self._h:
            lib().ss_destroy(self._h)
            self._h = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


_ctx_cache = {}


def default_context(device: int) -> Context:
    c = _ctx_cache.get(device)
    if c is None:
        c = _ctx_cache[device] = Context(device)
    return c


def _stream_ptr(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return _vp(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dtype_code(t):
    import torch
    if t.dtype == torch.float32:
        return SS_F32
    if t.dtype == torch.bfloat16:
        return SS_BF16
    raise TypeError("expected float32 or bfloat16, got %s" % t.dtype)


def _p(t):
    return None if t is None else _vp(t.data_ptr())


def _need(t, name, shape=None, dtype=None, device=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s has dtype %s, expected %s" % (name, t.dtype, dtype))
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))


def ss_scan_fwd(u, delta, A, B, C, D=None, delta_bias=None, z=None, delta_softplus=True,
                h0=None, y=None, h_last=None, out_dtype=None, return_last_state=True,
                ctx: Context | None = None, stream=None):
    """Selective scan forward on the GPU.

    u, delta, z: (batch, dim, L), B, C: (batch, N, L), all float32 or all
    bfloat16. A: (dim, N) float32; D, delta_bias: (dim,) float32 or None;
    h0: (batch, dim, N) float32 or None. y (batch, dim, L) and h_last
    (batch, dim, N) are allocated when not given; y defaults to float32.
    Returns (y, h_last) (h_last None when return_last_state is False and no
    buffer was given). Asynchronous on the current stream."""
    import torch
    _need(u, "u")
    batch, dim, L = u.shape
    N = B.shape[1]
    dev = u.device
    _need(delta, "delta", u.shape, u.dtype, dev)
    if z is not None:
        _need(z, "z", u.shape, u.dtype, dev)
    _need(B, "B", (batch, N, L), u.dtype, dev)
    _need(C, "C", (batch, N, L), u.dtype, dev)
    _need(A, "A", (dim, N), torch.float32, dev)
    if D is not None:
        _need(D, "D", (dim,), torch.float32, dev)
    if delta_bias is not None:
        _need(delta_bias, "delta_bias", (dim,), torch.float32, dev)
    if h0 is not None:
        _need(h0, "h0", (batch, dim, N), torch.float32, dev)
    if y is None:
        y = torch.empty((batch, dim, L), dtype=out_dtype or torch.float32, device=dev)
    _need(y, "y", (batch, dim, L), None, dev)
    if h_last is None and return_last_state:
        h_last = torch.empty((batch, dim, N), dtype=torch.float32, device=dev)
    if h_last is not None:
        _need(h_last, "h_last", (batch, dim, N), torch.float32, dev)
    a = ScanArgs(batch, dim, N, L, _dtype_code(u), _dtype_code(y), _p(u), _p(delta), _p(z),
                 _p(A), _p(B), _p(C), _p(D), _p(delta_bias), int(bool(delta_softplus)), _p(h0),
                 _p(y), _p(h_last))
    ctx = ctx or default_context(dev.index if dev.index is not None else 0)
    _check(lib().ss_scan_fwd(ctx.handle, ctypes.byref(a), _stream_ptr(stream, dev)),
           "ss_scan_fwd")
    return y, h_last


class PreparedScan:
    """An ss_scan_fwd call whose arguments were checked and marshalled once.

    Calling it enqueues the same scan again (same tensors, context and
    stream), with none of the per-call Python checks; for loops that run one
    shape over buffers that stay in place. The tensors must outlive it."""

    def __init__(self, u, delta, A, B, C, D=None, delta_bias=None, z=None, delta_softplus=True,
                 h0=None, y=None, h_last=None, out_dtype=None, ctx: Context | None = None,
                 stream=None):
        import torch
        self.y, self.h_last = y, h_last
        # the one-time checks are those of ss_scan_fwd; allocate outputs the same way
        _need(u, "u")
        batch, dim, L = u.shape
        N = B.shape[1]
        dev = u.device
        _need(delta, "delta", u.shape, u.dtype, dev)
        if z is not None:
            _need(z, "z", u.shape, u.dtype, dev)
        _need(B, "B", (batch, N, L), u.dtype, dev)
        _need(C, "C", (batch, N, L), u.dtype, dev)
        _need(A, "A", (dim, N), torch.float32, dev)
        for t, name in ((D, "D"), (delta_bias, "delta_bias")):
            if t is not None:
                _need(t, name, (dim,), torch.float32, dev)
        if h0 is not None:
            _need(h0, "h0", (batch, dim, N), torch.float32, dev)
        if self.y is None:
            self.y = torch.empty((batch, dim, L), dtype=out_dtype or torch.float32, device=dev)
        _need(self.y, "y", (batch, dim, L), None, dev)
        if self.h_last is not None:
            _need(self.h_last, "h_last", (batch, dim, N), torch.float32, dev)
        self._keep = (u, delta, A, B, C, D, delta_bias, z, h0)
        self._args = ScanArgs(batch, dim, N, L, _dtype_code(u), _dtype_code(self.y), _p(u),
                              _p(delta), _p(z), _p(A), _p(B), _p(C), _p(D), _p(delta_bias),
                              int(bool(delta_softplus)), _p(h0), _p(self.y), _p(self.h_last))
        self.ctx = ctx or default_context(dev.index if dev.index is not None else 0)
        self._stream = _stream_ptr(stream, dev)
        self._fn = lib().ss_scan_fwd
        self._argp = ctypes.byref(self._args)

    def __call__(self):
        rc = self._fn(self.ctx.handle, self._argp, self._stream)
        if rc != SS_OK:
            raise SSError(rc, "ss_scan_fwd")
        return self.y, self.h_last


def _conv_scan_args(x, conv_weight, delta, A, B, C, conv_bias, conv_init, conv_silu, D,
                    delta_bias, z, delta_softplus, h0, y, h_last, out_dtype, u_out,
                    conv_state_out, want_u, want_conv_state):
    """Checks and marshals the arguments of ss_conv_scan_fwd; allocates the
    outputs that were asked for but not given."""
    import torch
    _need(x, "x")
    batch, dim, L = x.shape
    N = B.shape[1]
    dev = x.device
    _need(conv_weight, "conv_weight", None, torch.float32, dev)
    if conv_weight.dim() != 2 or conv_weight.shape[0] != dim:
        raise ValueError("conv_weight must be (dim, width)")
    W = conv_weight.shape[1]
    _need(delta, "delta", x.shape, x.dtype, dev)
    if z is not None:
        _need(z, "z", x.shape, x.dtype, dev)
    _need(B, "B", (batch, N, L), x.dtype, dev)
    _need(C, "C", (batch, N, L), x.dtype, dev)
    _need(A, "A", (dim, N), torch.float32, dev)
    for t, name in ((D, "D"), (delta_bias, "delta_bias"), (conv_bias, "conv_bias")):
        if t is not None:
            _need(t, name, (dim,), torch.float32, dev)
    if conv_init is not None:
        _need(conv_init, "conv_init", (batch, dim, W - 1), torch.float32, dev)
    if h0 is not None:
        _need(h0, "h0", (batch, dim, N), torch.float32, dev)
    if y is None:
        y = torch.empty((batch, dim, L), dtype=out_dtype or torch.float32, device=dev)
    _need(y, "y", (batch, dim, L), None, dev)
    if h_last is None:
        h_last = torch.empty((batch, dim, N), dtype=torch.float32, device=dev)
    _need(h_last, "h_last", (batch, dim, N), torch.float32, dev)
    if u_out is None and want_u:
        u_out = torch.empty((batch, dim, L), dtype=x.dtype, device=dev)
    if u_out is not None:
        _need(u_out, "u_out", x.shape, x.dtype, dev)
    if conv_state_out is None and want_conv_state:
        conv_state_out = torch.empty((batch, dim, W - 1), dtype=torch.float32, device=dev)
    if conv_state_out is not None:
        _need(conv_state_out, "conv_state_out", (batch, dim, W - 1), torch.float32, dev)
    scan = ScanArgs(batch, dim, N, L, _dtype_code(x), _dtype_code(y), _p(x), _p(delta), _p(z),
                    _p(A), _p(B), _p(C), _p(D), _p(delta_bias), int(bool(delta_softplus)),
                    _p(h0), _p(y), _p(h_last))
    a = ConvScanArgs(scan, W, _p(conv_weight), _p(conv_bias), _p(conv_init), int(bool(conv_silu)),
                     _p(u_out), _p(conv_state_out))
    keep = (x, conv_weight, delta, A, B, C, conv_bias, conv_init, D, delta_bias, z, h0)
    return a, dev, (y, h_last, u_out, conv_state_out), keep


def ss_conv_scan_fwd(x, conv_weight, delta, A, B, C, conv_bias=None, conv_init=None,
                     conv_silu=True, D=None, delta_bias=None, z=None, delta_softplus=True,
                     h0=None, y=None, h_last=None, out_dtype=None, u_out=None,
                     conv_state_out=None, return_u=False, return_conv_state=False,
                     ctx: Context | None = None, stream=None):
    """The Mamba block's causal conv1d fused in front of the selective scan.

    x (the convolution's input), delta, z: (batch, dim, L); B, C: (batch, N, L);
    conv_weight (dim, width) float32, width 2..4; conv_bias (dim,) and
    conv_init (batch, dim, width-1) float32 or None. u = silu(conv(x)) (conv(x)
    when conv_silu is False) feeds the scan as in ss_scan_fwd. Returns
    (y, h_last, u_out, conv_state_out): the last two are None unless given or
    asked for with return_u / return_conv_state. Asynchronous."""
    a, dev, outs, _ = _conv_scan_args(x, conv_weight, delta, A, B, C, conv_bias, conv_init,
                                      conv_silu, D, delta_bias, z, delta_softplus, h0, y, h_last,
                                      out_dtype, u_out, conv_state_out, return_u,
                                      return_conv_state)
    ctx = ctx or default_context(dev.index if dev.index is not None else 0)
    _check(lib().ss_conv_scan_fwd(ctx.handle, ctypes.byref(a), _stream_ptr(stream, dev)),
           "ss_conv_scan_fwd")
    return outs


class PreparedConvScan:
    """An ss_conv_scan_fwd call whose arguments were checked and marshalled
    once (see PreparedScan); outputs are held in .outputs."""

    def __init__(self, x, conv_weight, delta, A, B, C, ctx: Context | None = None, stream=None,
                 **kw):
        args = dict(conv_bias=None, conv_init=None, conv_silu=True, D=None, delta_bias=None,
                    z=None, delta_softplus=True, h0=None, y=None, h_last=None, out_dtype=None,
                    u_out=None, conv_state_out=None, return_u=False, return_conv_state=False)
        args.update(kw)
        self._args, dev, self.outputs, self._keep = _conv_scan_args(
            x, conv_weight, delta, A, B, C, args["conv_bias"], args["conv_init"],
            args["conv_silu"], args["D"], args["delta_bias"], args["z"], args["delta_softplus"],
            args["h0"], args["y"], args["h_last"], args["out_dtype"], args["u_out"],
            args["conv_state_out"], args["return_u"], args["return_conv_state"])
        self.ctx = ctx or default_context(dev.index if dev.index is not None else 0)
        self._stream = _stream_ptr(stream, dev)
        self._fn = lib().ss_conv_scan_fwd
        self._argp = ctypes.byref(self._args)

    def __call__(self):
        rc = self._fn(self.ctx.handle, self._argp, self._stream)
        if rc != SS_OK:
            raise SSError(rc, "ss_conv_scan_fwd")
        return self.outputs


def ss_state_update(state, x, dt, A, B, C, D=None, dt_bias=None, z=None, dt_softplus=True,
                    y=None, out_dtype=None, ctx: Context | None = None, stream=None):
    """One decode step on the GPU; `state` (batch, dim, N) float32 is updated
    in place. x, dt, z: (batch, dim); B, C: (batch, N); A: (dim, N) float32.
    Returns y (batch, dim), float32 unless out_dtype/y say otherwise."""
    import torch
    _need(state, "state", None, torch.float32)
    batch, dim, N = state.shape
    dev = state.device
    _need(x, "x", (batch, dim), None, dev)
    _need(dt, "dt", (batch, dim), x.dtype, dev)
    if z is not None:
        _need(z, "z", (batch, dim), x.dtype, dev)
    _need(B, "B", (batch, N), x.dtype, dev)
    _need(C, "C", (batch, N), x.dtype, dev)
    _need(A, "A", (dim, N), torch.float32, dev)
    if D is not None:
        _need(D, "D", (dim,), torch.float32, dev)
    if dt_bias is not None:
        _need(dt_bias, "dt_bias", (dim,), torch.float32, dev)
    if y is None:
        y = torch.empty((batch, dim), dtype=out_dtype or torch.float32, device=dev)
    _need(y, "y", (batch, dim), None, dev)
    a = UpdateArgs(batch, dim, N, _dtype_code(x), _dtype_code(y), _p(state), _p(x), _p(dt),
                   _p(z), _p(A), _p(B), _p(C), _p(D), _p(dt_bias), int(bool(dt_softplus)), _p(y))
    ctx = ctx or default_context(dev.index if dev.index is not None else 0)
    _check(lib().ss_state_update(ctx.handle, ctypes.byref(a), _stream_ptr(stream, dev)),
           "ss_state_update")
    return y


def ss_scan_bwd(u, delta, A, B, C, dy, D=None, delta_bias=None, z=None, delta_softplus=True,
                h0=None, dh_last=None, ctx: Context | None = None, stream=None):
    """Gradients of the selective scan on the GPU.

    Inputs as for ss_scan_fwd; dy (batch, dim, L) and dh_last (batch, dim, N)
    float32 (dh_last may be None). Returns a dict of float32 tensors: du,
    ddelta, dz (None without z), dA, dB, dC, dD (None without D), ddelta_bias
    (None without delta_bias), dh0 (None without h0)."""
    import torch
    _need(u, "u")
    batch, dim, L = u.shape
    N = B.shape[1]
    dev = u.device
    _need(delta, "delta", u.shape, u.dtype, dev)
    if z is not None:
        _need(z, "z", u.shape, u.dtype, dev)
    _need(B, "B", (batch, N, L), u.dtype, dev)
    _need(C, "C", (batch, N, L), u.dtype, dev)
    _need(A, "A", (dim, N), torch.float32, dev)
    for t, name in ((D, "D"), (delta_bias, "delta_bias")):
        if t is not None:
            _need(t, name, (dim,), torch.float32, dev)
    if h0 is not None:
        _need(h0, "h0", (batch, dim, N), torch.float32, dev)
    _need(dy, "dy", (batch, dim, L), torch.float32, dev)
    if dh_last is not None:
        _need(dh_last, "dh_last", (batch, dim, N), torch.float32, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    g = dict(du=torch.empty((batch, dim, L), **f32), ddelta=torch.empty((batch, dim, L), **f32),
             dz=torch.empty((batch, dim, L), **f32) if z is not None else None,
             dA=torch.empty((dim, N), **f32), dB=torch.empty((batch, N, L), **f32),
             dC=torch.empty((batch, N, L), **f32),
             dD=torch.empty((dim,), **f32) if D is not None else None,
             ddelta_bias=torch.empty((dim,), **f32) if delta_bias is not None else None,
             dh0=torch.empty((batch, dim, N), **f32) if h0 is not None else None)
    a = ScanBwdArgs(batch, dim, N, L, _dtype_code(u), _p(u), _p(delta), _p(z), _p(A), _p(B),
                    _p(C), _p(D), _p(delta_bias), int(bool(delta_softplus)), _p(h0), _p(dy),
                    _p(dh_last), _p(g["du"]), _p(g["ddelta"]), _p(g["dz"]), _p(g["dA"]),
                    _p(g["dB"]), _p(g["dC"]), _p(g["dD"]), _p(g["ddelta_bias"]), _p(g["dh0"]))
    ctx = ctx or default_context(dev.index if dev.index is not None else 0)
    _check(lib().ss_scan_bwd(ctx.handle, ctypes.byref(a), _stream_ptr(stream, dev)),
           "ss_scan_bwd")
    return g


def ss_ssd_fwd(x, dt, A, B, C, D=None, dt_bias=None, dt_softplus=True, h0=None, y=None,
               h_last=None, out_dtype=None, return_last_state=True, ctx: Context | None = None,
               stream=None):
    """Mamba-2 SSD forward on the GPU (chunked, tensor-core products).

    x (batch, L, heads, headdim) bfloat16; dt (batch, L, heads) bfloat16;
    A (heads,) float32; B, C (batch, L, dstate) bfloat16; D, dt_bias (heads,)
    float32 or None; h0 (batch, heads, headdim, dstate) float32 or None.
    Returns (y, h_last); y defaults to float32."""
    import torch
    _need(x, "x")
    batch, L, H, P = x.shape
    N = B.shape[2]
    dev = x.device
    _need(dt, "dt", (batch, L, H), x.dtype, dev)
    _need(A, "A", (H,), torch.float32, dev)
    _need(B, "B", (batch, L, N), x.dtype, dev)
    _need(C, "C", (batch, L, N), x.dtype, dev)
    for t, name in ((D, "D"), (dt_bias, "dt_bias")):
        if t is not None:
            _need(t, name, (H,), torch.float32, dev)
    if h0 is not None:
        _need(h0, "h0", (batch, H, P, N), torch.float32, dev)
    if y is None:
        y = torch.empty((batch, L, H, P), dtype=out_dtype or torch.float32, device=dev)
    _need(y, "y", (batch, L, H, P), None, dev)
    if h_last is None and return_last_state:
        h_last = torch.empty((batch, H, P, N), dtype=torch.float32, device=dev)
    if h_last is not None:
        _need(h_last, "h_last", (batch, H, P, N), torch.float32, dev)
    a = SsdArgs(batch, H, P, N, L, _dtype_code(x), _dtype_code(y), _p(x), _p(dt), _p(A), _p(B),
                _p(C), _p(D), _p(dt_bias), int(bool(dt_softplus)), _p(h0), _p(y), _p(h_last))
    ctx = ctx or default_context(dev.index if dev.index is not None else 0)
    _check(lib().ss_ssd_fwd(ctx.handle, ctypes.byref(a), _stream_ptr(stream, dev)), "ss_ssd_fwd")
    return y, h_last


def ss_conv1d_fwd(x, weight, bias=None, init_state=None, silu=False, out=None,
                  final_state=None, out_dtype=None, return_final_state=True,
                  ctx: Context | None = None, stream=None):
    """Causal depthwise convolution on the GPU.

    x (batch, dim, L) float32 or bfloat16; weight (dim, W) float32 with W in
    {2, 3, 4}; bias (dim,) float32 or None; init_state (batch, dim, W-1)
    float32 or None (the W-1 inputs before step 0, oldest first). out defaults
    to x's dtype. Returns (out, final_state), final_state (batch, dim, W-1)
    float32 (None when return_final_state is False and no buffer was given)."""
    import torch
    _need(x, "x")
    batch, dim, L = x.shape
    dev = x.device
    _need(weight, "weight", None, torch.float32, dev)
    if weight.dim() != 2 or weight.shape[0] != dim:
        raise ValueError("weight must be (dim, width)")
    W = weight.shape[1]
    if bias is not None:
        _need(bias, "bias", (dim,), torch.float32, dev)
    if init_state is not None:
        _need(init_state, "init_state", (batch, dim, W - 1), torch.float32, dev)
    if out is None:
        out = torch.empty((batch, dim, L), dtype=out_dtype or x.dtype, device=dev)
    _need(out, "out", (batch, dim, L), None, dev)
    if final_state is None and return_final_state:
        final_state = torch.empty((batch, dim, W - 1), dtype=torch.float32, device=dev)
    if final_state is not None:
        _need(final_state, "final_state", (batch, dim, W - 1), torch.float32, dev)
    a = Conv1dArgs(batch, dim, W, L, _dtype_code(x), _dtype_code(out), _p(x), _p(weight),
                   _p(bias), _p(init_state), int(bool(silu)), _p(out), _p(final_state))
    ctx = ctx or default_context(dev.index if dev.index is not None else 0)
    _check(lib().ss_conv1d_fwd(ctx.handle, ctypes.byref(a), _stream_ptr(stream, dev)),
           "ss_conv1d_fwd")
    return out, final_state


def ss_conv1d_update(state, x, weight, bias=None, silu=False, out=None, out_dtype=None,
                     ctx: Context | None = None, stream=None):
    """One decode step of the convolution; state (batch, dim, W-1) float32 is
    updated in place. x (batch, dim). Returns out (batch, dim), x's dtype
    unless out/out_dtype say otherwise."""
    import torch
    _need(state, "state", None, torch.float32)
    batch, dim, Wm1 = state.shape
    dev = state.device
    _need(x, "x", (batch, dim), None, dev)
    _need(weight, "weight", (dim, Wm1 + 1), torch.float32, dev)
    if bias is not None:
        _need(bias, "bias", (dim,), torch.float32, dev)
    if out is None:
        out = torch.empty((batch, dim), dtype=out_dtype or x.dtype, device=dev)
    _need(out, "out", (batch, dim), None, dev)
    a = Conv1dUpdateArgs(batch, dim, Wm1 + 1, _dtype_code(x), _dtype_code(out), _p(state),
                         _p(x), _p(weight), _p(bias), int(bool(silu)), _p(out))
    ctx = ctx or default_context(dev.index if dev.index is not None else 0)
    _check(lib().ss_conv1d_update(ctx.handle, ctypes.byref(a), _stream_ptr(stream, dev)),
           "ss_conv1d_update")
    return out


__all__ = ["ss_scan_fwd", "ss_scan_bwd", "ss_ssd_fwd", "ss_state_update", "ss_conv1d_fwd",
           "ss_conv1d_update",
           "PreparedScan", "Context", "SSError", "lib", "status_string",
           "ScanArgs", "UpdateArgs", "ScanBwdArgs", "SsdArgs", "Conv1dArgs", "Conv1dUpdateArgs",
           "LIB_PATH"]
