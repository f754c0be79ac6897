"""ctypes binding of libq8proj.so: argument marshalling only.

Every function here has the name of the C entry point it calls and does no
arithmetic of its own: it checks tensor dtypes/shapes/devices, passes raw
device pointers, sizes and the current CUDA stream, and turns a non-zero
status into :class:`Q8Error`.  If the library is missing the call fails
loudly; there is no CPU or PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

STATUS_NAMES = {0: "Q8_OK", 1: "Q8_ERR_ARG", 2: "Q8_ERR_ALIGN", 3: "Q8_ERR_DEVICE", 4: "Q8_ERR_LAUNCH",
                5: "Q8_ERR_DEVICE_TIMEOUT", 6: "Q8_ERR_CUDA", 7: "Q8_ERR_TOO_BIG"}

# (name, restype, argtypes) of every symbol include/q8proj.h declares.
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_INT = ctypes.c_int
SIGNATURES = {
    "q8_plane_rows": (_I64, [_I64]),
    "q8_strerror": (ctypes.c_char_p, [_INT]),
    "quantize_q8_0": (_INT, [_P, _I64, _I64, _P, _P, _I64, _P]),
    "rmsnorm_quant": (_INT, [_P, _P, ctypes.c_float, _P, _I64, _I64, _P, _P, _I64, _P]),
    "swiglu_quant": (_INT, [_P, _P, _P, _I64, _I64, _P, _P, _I64, _P]),
    "q8_0_gemv": (_INT, [_P, _I64, _I64, _P, _P, _P, _P]),
    "q8_0_gemm_workspace_bytes": (ctypes.c_size_t, [_I64, _I64, _I64]),
    "q8_0_gemm": (_INT, [_P, _I64, _I64, _P, _P, _I64, _I64, _P, _P, ctypes.c_size_t, _P]),
    "q8_0_gemm_prepared_weights_bytes": (ctypes.c_size_t, [_I64, _I64]),
    "q8_0_gemm_prepare_weights": (_INT, [_P, _I64, _I64, _P, ctypes.c_size_t, _P]),
    "q8_0_gemm_prepared_workspace_bytes": (ctypes.c_size_t, [_I64, _I64, _I64]),
    "q8_0_gemm_prepared": (_INT, [_P, _P, _I64, _I64, _P, _P, _I64, _I64, _P, _P, ctypes.c_size_t, _P]),
    "q8_0_gemm_mma": (_INT, [_P, _I64, _I64, _P, _P, _I64, _I64, _P, _P]),
    "q8_0_gemm_noalloc": (_INT, [_P, _I64, _I64, _P, _P, _I64, _I64, _P, _P]),
    "q8_0_gemm_noalloc_max_bytes": (ctypes.c_size_t, []),
    "q8_0_gemv_grouped": (_INT, [_P, _INT, _I64, _P, _P, _P]),
    "q8_0_gemv_fused": (_INT, [_P, _INT, _I64, _INT, _P, _P, _P, ctypes.c_float, _P]),
    "q8_0_gemv_gate_up": (_INT, [_P, _P, _I64, _I64, _P, _P, _INT, _P, _P, ctypes.c_float, _P, _P, _P, _P, _P]),
    "q8_0_gemv_batched": (_INT, [_P, _I64, _I64, _P, _P, _I64, _P, _P]),
    "q8_0_gemv_batched_grouped": (_INT, [_P, _INT, _I64, _P, _P, _I64, _P]),
    "q4a_gemv": (_INT, [_P, _I64, _I64, _P, _P, _P, _P]),
    "q4a_gemv_batched": (_INT, [_P, _I64, _I64, _P, _P, _I64, _P, _P]),
    "q4a_gemv_batched_grouped": (_INT, [_P, _INT, _I64, _P, _P, _I64, _P]),
    "q8_check": (_INT, [_P]),
    "q8_num_sms": (_INT, []),
}


MAX_GROUP = 8
GEMV_MAX_TOKENS = 16
PRODUCER_QUANT, PRODUCER_RMSNORM, PRODUCER_SWIGLU = 1, 2, 3


class GemvProj(ctypes.Structure):
    """C struct q8_gemv_proj: one projection of a grouped GEMV."""

    _fields_ = [("w", ctypes.c_void_p), ("n", ctypes.c_int64), ("y", ctypes.c_void_p)]


class Q8Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = lib().q8_strerror(status).decode() if _lib is not None else ""
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}: {msg}")


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libq8proj.so (built in-tree by ``build.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libq8proj.so is not built ({path}); run int8_quantized_projection_gb300.build")
            h = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(h, name)
                f.restype = res
                f.argtypes = args
            _lib = h
        return _lib


def load():
    return lib()


def _stream(stream):
    if stream is None:
        import torch

        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _check(fn, st):
    if st != 0:
        raise Q8Error(fn, st)


class Bound:
    """A C entry point with its arguments already marshalled.

    Calling it re-issues the same launch (same pointers, sizes and stream)
    with one ctypes call, which keeps the host cost of a decode step far below
    the GPU time of its kernels.  Returned by the ``bind=True`` form of every
    launching function."""

    __slots__ = ("name", "fn", "args", "_keep")

    def __init__(self, name, args):
        self.name = name
        self.fn = getattr(lib(), name)
        self.args = args
        self._keep = None

    def __call__(self):
        st = self.fn(*self.args)
        if st != 0:
            raise Q8Error(self.name, st)


def _launch(name, args, bind):
    if bind:
        return Bound(name, args)
    _check(name, getattr(lib(), name)(*args))
    return None


def _need(t, dtype, name):
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous CUDA tensor of {dtype}, got {t.dtype} on {t.device}")


def q8_plane_rows(rows: int) -> int:
    return int(lib().q8_plane_rows(rows))


def q8_num_sms() -> int:
    return int(lib().q8_num_sms())


def q8_check(stream=None) -> None:
    _check("q8_check", lib().q8_check(_stream(stream)))


def quantize_q8_0(x, qs, ds, stream=None, bind=False):
    """x f32 [rows][k] -> plane (qs int8 [rows_pad][k], ds int32 [rows_pad][k/32])."""
    import torch

    _need(x, torch.float32, "x"), _need(qs, torch.int8, "qs"), _need(ds, torch.int32, "ds")
    rows, k = x.shape
    rows_pad = qs.shape[0]
    if qs.shape != (rows_pad, k) or ds.shape != (rows_pad, k // 32):
        raise ValueError("plane shape mismatch")
    return _launch("quantize_q8_0", (_ptr(x), rows, k, _ptr(qs), _ptr(ds), rows_pad, _stream(stream)), bind)


def rmsnorm_quant(x, w, eps: float, y, qs, ds, stream=None, bind=False):
    """``y=None``: mode 2, only the plane is written (the f32 output is dead)."""
    import torch

    for t, n in ((x, "x"), (w, "w")) + (((y, "y"),) if y is not None else ()):
        _need(t, torch.float32, n)
    _need(qs, torch.int8, "qs"), _need(ds, torch.int32, "ds")
    rows, d = x.shape
    rows_pad = qs.shape[0]
    if ((y is not None and y.shape != x.shape) or w.shape != (d,) or qs.shape != (rows_pad, d)
            or ds.shape != (rows_pad, d // 32)):
        raise ValueError("shape mismatch")
    yp = _ptr(y) if y is not None else ctypes.c_void_p(0)
    return _launch("rmsnorm_quant", (_ptr(x), _ptr(w), ctypes.c_float(eps), yp, rows, d, _ptr(qs), _ptr(ds),
                                     rows_pad, _stream(stream)), bind)


def swiglu_quant(gate, up, y, qs, ds, stream=None, bind=False):
    """``y=None``: mode 2, only the plane is written (the f32 output is dead)."""
    import torch

    for t, n in ((gate, "gate"), (up, "up")) + (((y, "y"),) if y is not None else ()):
        _need(t, torch.float32, n)
    _need(qs, torch.int8, "qs"), _need(ds, torch.int32, "ds")
    rows, nf = gate.shape
    rows_pad = qs.shape[0]
    if (up.shape != gate.shape or (y is not None and y.shape != gate.shape) or qs.shape != (rows_pad, nf)
            or ds.shape != (rows_pad, nf // 32)):
        raise ValueError("shape mismatch")
    yp = _ptr(y) if y is not None else ctypes.c_void_p(0)
    return _launch("swiglu_quant", (_ptr(gate), _ptr(up), yp, rows, nf, _ptr(qs), _ptr(ds), rows_pad,
                                    _stream(stream)), bind)


def q8_0_gemv(w, n: int, k: int, qs, ds, y, stream=None, bind=False):
    """w uint8 [n*k/32*34] Q8_0 blocks; plane row 0 of (qs, ds); y f32 [n]."""
    import torch

    _need(w, torch.uint8, "w"), _need(qs, torch.int8, "qs"), _need(ds, torch.int32, "ds"), _need(y, torch.float32, "y")
    if w.numel() != n * (k // 32) * 34 or y.numel() < n or qs.shape[-1] != k:
        raise ValueError("shape mismatch")
    return _launch("q8_0_gemv", (_ptr(w), n, k, _ptr(qs), _ptr(ds), _ptr(y), _stream(stream)), bind)


def q8_0_gemv_batched(w, n: int, k: int, qs, ds, t: int, y, stream=None, bind=False):
    """Y[t][n] f32 for plane rows [0, t), 1 <= t <= 16, weights read once for all t."""
    import torch

    _need(w, torch.uint8, "w"), _need(qs, torch.int8, "qs"), _need(ds, torch.int32, "ds"), _need(y, torch.float32, "y")
    if w.numel() != n * (k // 32) * 34 or y.numel() < t * n or qs.shape[-1] != k or qs.shape[0] < t:
        raise ValueError("shape mismatch")
    return _launch("q8_0_gemv_batched", (_ptr(w), n, k, _ptr(qs), _ptr(ds), t, _ptr(y), _stream(stream)), bind)


def q8_0_gemv_batched_grouped(projs, k: int, qs, ds, t: int, stream=None, bind=False):
    """Several small-batch projections of the same plane rows [0, t) in one launch.

    ``projs`` is a sequence of (w uint8 Q8_0 blocks, n, y f32 [t][n]) sharing k."""
    import torch

    _need(qs, torch.int8, "qs"), _need(ds, torch.int32, "ds")
    if not 1 <= len(projs) <= MAX_GROUP or qs.shape[-1] != k or qs.shape[0] < t:
        raise ValueError("1..8 projections sharing k and the plane")
    arr = (GemvProj * len(projs))()
    keep = []
    for i, (w, n, y) in enumerate(projs):
        _need(w, torch.uint8, "w"), _need(y, torch.float32, "y")
        if w.numel() != n * (k // 32) * 34 or y.numel() < t * n:
            raise ValueError("shape mismatch")
        arr[i] = GemvProj(w.data_ptr(), n, y.data_ptr())
        keep.append((w, y))
    args = (ctypes.cast(arr, ctypes.c_void_p), len(projs), k, _ptr(qs), _ptr(ds), t, _stream(stream))
    if bind:
        b = Bound("q8_0_gemv_batched_grouped", args)
        b._keep = (arr, keep)  # the descriptor array must outlive the bound launch
        return b
    _check("q8_0_gemv_batched_grouped", lib().q8_0_gemv_batched_grouped(*args))
    return None


def q4a_gemv(w, n: int, k: int, qs, ds, y, stream=None, bind=False):
    """w uint8 [n*k/32*20] asymmetric 4-bit blocks; plane row 0 of (qs, ds); y f32 [n]."""
    import torch

    _need(w, torch.uint8, "w"), _need(qs, torch.int8, "qs"), _need(ds, torch.int32, "ds"), _need(y, torch.float32, "y")
    if w.numel() != n * (k // 32) * 20 or y.numel() < n or qs.shape[-1] != k:
        raise ValueError("shape mismatch")
    return _launch("q4a_gemv", (_ptr(w), n, k, _ptr(qs), _ptr(ds), _ptr(y), _stream(stream)), bind)


def q4a_gemv_batched(w, n: int, k: int, qs, ds, t: int, y, stream=None, bind=False):
    """Asymmetric 4-bit weights, Y[t][n] f32 for plane rows [0, t), 1 <= t <= 16, weights read once for all t."""
    import torch

    _need(w, torch.uint8, "w"), _need(qs, torch.int8, "qs"), _need(ds, torch.int32, "ds"), _need(y, torch.float32, "y")
    if w.numel() != n * (k // 32) * 20 or y.numel() < t * n or qs.shape[-1] != k or qs.shape[0] < t:
        raise ValueError("shape mismatch")
    return _launch("q4a_gemv_batched", (_ptr(w), n, k, _ptr(qs), _ptr(ds), t, _ptr(y), _stream(stream)), bind)


def q4a_gemv_batched_grouped(projs, k: int, qs, ds, t: int, stream=None, bind=False):
    """Several asymmetric 4-bit small-batch projections of the same plane rows [0, t) in one launch.

    ``projs`` is a sequence of (w uint8 20-byte blocks, n, y f32 [t][n]) sharing k."""
    import torch

    _need(qs, torch.int8, "qs"), _need(ds, torch.int32, "ds")
    if not 1 <= len(projs) <= MAX_GROUP or qs.shape[-1] != k or qs.shape[0] < t:
        raise ValueError("1..8 projections sharing k and the plane")
    arr = (GemvProj * len(projs))()
    keep = []
    for i, (w, n, y) in enumerate(projs):
        _need(w, torch.uint8, "w"), _need(y, torch.float32, "y")
        if w.numel() != n * (k // 32) * 20 or y.numel() < t * n:
            raise ValueError("shape mismatch")
        arr[i] = GemvProj(w.data_ptr(), n, y.data_ptr())
        keep.append((w, y))
    args = (ctypes.cast(arr, ctypes.c_void_p), len(projs), k, _ptr(qs), _ptr(ds), t, _stream(stream))
    if bind:
        b = Bound("q4a_gemv_batched_grouped", args)
        b._keep = (arr, keep)  # the descriptor array must outlive the bound launch
        return b
    _check("q4a_gemv_batched_grouped", lib().q4a_gemv_batched_grouped(*args))
    return None


def q8_0_gemv_grouped(projs, k: int, qs, ds, stream=None, bind=False):
    """Several projections of one activation in one launch.

    ``projs`` is a sequence of (w uint8 Q8_0 blocks, n, y f32 [n]) sharing k and
    plane row 0 of (qs, ds)."""
    import torch

    _need(qs, torch.int8, "qs"), _need(ds, torch.int32, "ds")
    if not 1 <= len(projs) <= MAX_GROUP or qs.shape[-1] != k:
        raise ValueError("1..8 projections sharing k")
    arr = (GemvProj * len(projs))()
    keep = []
    for i, (w, n, y) in enumerate(projs):
        _need(w, torch.uint8, "w"), _need(y, torch.float32, "y")
        if w.numel() != n * (k // 32) * 34 or y.numel() < n:
            raise ValueError("shape mismatch")
        arr[i] = GemvProj(w.data_ptr(), n, y.data_ptr())
        keep.append((w, y))
    args = (ctypes.cast(arr, ctypes.c_void_p), len(projs), k, _ptr(qs), _ptr(ds), _stream(stream))
    if bind:
        b = Bound("q8_0_gemv_grouped", args)
        b._keep = (arr, keep)  # the descriptor array must outlive the bound launch
        return b
    _check("q8_0_gemv_grouped", lib().q8_0_gemv_grouped(*args))
    return None


def _proj_array(projs, k):
    import torch

    if not 1 <= len(projs) <= MAX_GROUP:
        raise ValueError("1..8 projections sharing k")
    arr = (GemvProj * len(projs))()
    keep = []
    for i, (w, n, y) in enumerate(projs):
        _need(w, torch.uint8, "w"), _need(y, torch.float32, "y")
        if w.numel() != n * (k // 32) * 34 or y.numel() < n:
            raise ValueError("shape mismatch")
        arr[i] = GemvProj(w.data_ptr(), n, y.data_ptr())
        keep.append((w, y))
    return arr, keep


def q8_0_gemv_fused(projs, k: int, producer: int, a, b=None, norm_w=None, eps: float = 0.0, stream=None,
                    bind=False):
    """Grouped batch-1 projections whose activation the same launch produces.

    ``producer`` is PRODUCER_QUANT (a = x f32 [k]), PRODUCER_RMSNORM (a = x,
    norm_w = w f32 [k], eps) or PRODUCER_SWIGLU (a = gate, b = up, f32 [k]);
    ``projs`` as for :func:`q8_0_gemv_grouped`."""
    import torch

    for t, nm in ((a, "a"), (b, "b"), (norm_w, "norm_w")):
        if t is not None:
            _need(t, torch.float32, nm)
            if t.numel() < k:
                raise ValueError(f"{nm}: fewer than k elements")
    arr, keep = _proj_array(projs, k)
    nul = ctypes.c_void_p(0)
    args = (ctypes.cast(arr, ctypes.c_void_p), len(projs), k, int(producer), _ptr(a),
            _ptr(b) if b is not None else nul, _ptr(norm_w) if norm_w is not None else nul, float(eps),
            _stream(stream))
    if bind:
        bd = Bound("q8_0_gemv_fused", args)
        bd._keep = (arr, keep, a, b, norm_w)
        return bd
    _check("q8_0_gemv_fused", lib().q8_0_gemv_fused(*args))
    return None


def q8_0_gemv_gate_up(w_gate, w_up, nf: int, k: int, qs_out, ds_out, qs=None, ds=None, producer: int = 0, a=None,
                      norm_w=None, eps: float = 0.0, y_gate=None, y_up=None, stream=None, bind=False):
    """Gate and up projections of one token with SwiGLU + q8_0 quantize in the same launch.

    The activation is plane row 0 of (qs, ds) when ``producer`` is 0, else
    produced in the launch (PRODUCER_QUANT: a = x; PRODUCER_RMSNORM: a = x,
    norm_w, eps).  Writes plane row 0 of silu(gate) * up into (qs_out,
    ds_out); y_gate / y_up (f32 [nf]) are optional."""
    import torch

    _need(w_gate, torch.uint8, "w_gate"), _need(w_up, torch.uint8, "w_up")
    _need(qs_out, torch.int8, "qs_out"), _need(ds_out, torch.int32, "ds_out")
    if w_gate.numel() != nf * (k // 32) * 34 or w_up.numel() != w_gate.numel():
        raise ValueError("weight shape mismatch")
    if qs_out.shape[-1] != nf or ds_out.shape[-1] != nf // 32:
        raise ValueError("output plane shape mismatch")
    for t, nm, dt in ((qs, "qs", torch.int8), (ds, "ds", torch.int32), (a, "a", torch.float32),
                      (norm_w, "norm_w", torch.float32), (y_gate, "y_gate", torch.float32),
                      (y_up, "y_up", torch.float32)):
        if t is not None:
            _need(t, dt, nm)
    nul = ctypes.c_void_p(0)
    opt = lambda t: _ptr(t) if t is not None else nul  # noqa: E731
    args = (_ptr(w_gate), _ptr(w_up), nf, k, opt(qs), opt(ds), int(producer), opt(a), opt(norm_w), float(eps),
            opt(y_gate), opt(y_up), _ptr(qs_out), _ptr(ds_out), _stream(stream))
    return _launch("q8_0_gemv_gate_up", args, bind)


def q8_0_gemm_workspace_bytes(n: int, t: int, k: int) -> int:
    return int(lib().q8_0_gemm_workspace_bytes(n, t, k))


def gemm_workspace(n: int, t: int, k: int, device="cuda"):
    """Allocate (with PyTorch) the scratch q8_0_gemm needs for (t, k); None if it needs none."""
    import torch

    nbytes = q8_0_gemm_workspace_bytes(n, t, k)
    return torch.empty(nbytes, dtype=torch.uint8, device=device) if nbytes else None


def q8_0_gemm_prepared_weights_bytes(n: int, k: int) -> int:
    return int(lib().q8_0_gemm_prepared_weights_bytes(n, k))


def q8_0_gemm_prepared_workspace_bytes(n: int, t: int, k: int) -> int:
    return int(lib().q8_0_gemm_prepared_workspace_bytes(n, t, k))


def q8_0_gemm_prepare_weights(w, n: int, k: int, wprep=None, stream=None):
    """Write the GEMM's prepared form of the Q8_0 matrix ``w`` (n x k) into
    ``wprep`` (a uint8 CUDA tensor of q8_0_gemm_prepared_weights_bytes(n, k)
    bytes; allocated here with PyTorch when None) and return it."""
    import torch

    _need(w, torch.uint8, "w")
    if w.numel() != n * (k // 32) * 34:
        raise ValueError("shape mismatch")
    nbytes = q8_0_gemm_prepared_weights_bytes(n, k)
    if nbytes == 0:
        raise ValueError("no prepared form for this shape ((k/32) % 8 != 0 or past the GEMM's limits)")
    if wprep is None:
        wprep = torch.empty(nbytes, dtype=torch.uint8, device=w.device)
    _need(wprep, torch.uint8, "wprep")
    _check("q8_0_gemm_prepare_weights",
           lib().q8_0_gemm_prepare_weights(_ptr(w), n, k, _ptr(wprep), wprep.numel(), _stream(stream)))
    return wprep


def q8_0_gemm_prepared(w, wprep, n: int, k: int, qs, ds, t: int, y, workspace=None, stream=None, bind=False):
    """q8_0_gemm whose tcgen05 path reads ``wprep`` (q8_0_gemm_prepare_weights's
    output) instead of widening ``w`` on every call; ``w`` serves the other
    paths (t <= 64, (k/32) % 8 != 0) and may be None when the call takes the
    tcgen05 path."""
    import torch

    _need(qs, torch.int8, "qs"), _need(ds, torch.int32, "ds"), _need(y, torch.float32, "y")
    if w is not None:
        _need(w, torch.uint8, "w")
    if wprep is not None:
        _need(wprep, torch.uint8, "wprep")
    rows_pad = qs.shape[0]
    if y.numel() < t * n or qs.shape[-1] != k or ds.shape[0] != rows_pad:
        raise ValueError("shape mismatch")
    nbytes = q8_0_gemm_prepared_workspace_bytes(n, t, k)
    if workspace is None and nbytes:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=y.device)
    if workspace is not None:
        _need(workspace, torch.uint8, "workspace")
    nul = ctypes.c_void_p(0)
    args = (_ptr(w) if w is not None else nul, _ptr(wprep) if wprep is not None else nul, n, k, _ptr(qs), _ptr(ds),
            t, rows_pad, _ptr(y), _ptr(workspace) if workspace is not None else nul,
            workspace.numel() if workspace is not None else 0, _stream(stream))
    if bind:
        b = Bound("q8_0_gemm_prepared", args)
        b._keep = (workspace, w, wprep)
        return b
    _check("q8_0_gemm_prepared", lib().q8_0_gemm_prepared(*args))
    return None


def q8_0_gemm(w, n: int, k: int, qs, ds, t: int, y, workspace=None, stream=None, bind=False):
    """Y[t][n] f32 = plane rows [0, t) x Q8_0 weights.

    ``workspace`` is a uint8 CUDA tensor of at least q8_0_gemm_workspace_bytes(n, t, k)
    bytes; when None one is allocated here with PyTorch (the library never allocates)."""
    import torch

    _need(w, torch.uint8, "w"), _need(qs, torch.int8, "qs"), _need(ds, torch.int32, "ds"), _need(y, torch.float32, "y")
    rows_pad = qs.shape[0]
    if w.numel() != n * (k // 32) * 34 or y.numel() < t * n or qs.shape[-1] != k or ds.shape[0] != rows_pad:
        raise ValueError("shape mismatch")
    if workspace is None:
        workspace = gemm_workspace(n, t, k, y.device)
    if workspace is not None:
        _need(workspace, torch.uint8, "workspace")
    wsp = _ptr(workspace) if workspace is not None else ctypes.c_void_p(0)
    wsb = workspace.numel() if workspace is not None else 0
    args = (_ptr(w), n, k, _ptr(qs), _ptr(ds), t, rows_pad, _ptr(y), wsp, wsb, _stream(stream))
    if bind:
        b = Bound("q8_0_gemm", args)
        b._keep = workspace
        return b
    _check("q8_0_gemm", lib().q8_0_gemm(*args))
    return None


_noalloc_devices = set()  # devices on which an eager q8_0_gemm_noalloc call has succeeded


def q8_0_gemm_noalloc(w, n: int, k: int, qs, ds, t: int, y, stream=None, bind=False):
    """q8_0_gemm whose scratch is the library's fixed device array (no allocation anywhere).

    For callers that cannot allocate device memory here; requests larger than
    q8_0_gemm_noalloc_max_bytes() raise Q8Error(Q8_ERR_TOO_BIG).  Calls that overlap
    on the GPU share that array and race.  The first call on a device looks the
    array up (a host-side CUDA call), so ``bind=True`` -- the form used to record
    launches into a CUDA graph -- is refused until one eager call has been made on
    that device."""
    import torch

    _need(w, torch.uint8, "w"), _need(qs, torch.int8, "qs"), _need(ds, torch.int32, "ds"), _need(y, torch.float32, "y")
    rows_pad = qs.shape[0]
    if w.numel() != n * (k // 32) * 34 or y.numel() < t * n or qs.shape[-1] != k or ds.shape[0] != rows_pad:
        raise ValueError("shape mismatch")
    dev = y.device.index if y.device.index is not None else torch.cuda.current_device()
    if bind and dev not in _noalloc_devices:
        raise RuntimeError("q8_0_gemm_noalloc: make one eager call on this device before binding it (its first call "
                           "looks up the scratch array's device address, which must not happen inside a stream capture)")
    out = _launch("q8_0_gemm_noalloc", (_ptr(w), n, k, _ptr(qs), _ptr(ds), t, rows_pad, _ptr(y), _stream(stream)),
                  bind)
    if not bind:
        _noalloc_devices.add(dev)
    return out


def q8_0_gemm_mma(w, n: int, k: int, qs, ds, t: int, y, stream=None, bind=False):
    """Legacy-tensor-path A/B twin of :func:`q8_0_gemm` (mma.sync.m16n8k32.s8)."""
    import torch

    _need(w, torch.uint8, "w"), _need(qs, torch.int8, "qs"), _need(ds, torch.int32, "ds"), _need(y, torch.float32, "y")
    rows_pad = qs.shape[0]
    if w.numel() != n * (k // 32) * 34 or y.numel() < t * n or qs.shape[-1] != k or ds.shape[0] != rows_pad:
        raise ValueError("shape mismatch")
    return _launch("q8_0_gemm_mma", (_ptr(w), n, k, _ptr(qs), _ptr(ds), t, rows_pad, _ptr(y), _stream(stream)), bind)


def empty_plane(rows_pad: int, k: int, device="cuda"):
    """Allocate (with PyTorch) an uninitialised plane: (qs int8, ds int32)."""
    import torch

    return (torch.empty((rows_pad, k), dtype=torch.int8, device=device),
            torch.empty((rows_pad, k // 32), dtype=torch.int32, device=device))
