"""CPU oracle for the int8 quantized projection path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library
and its Python binding) never imports it, and it imports nothing from the
product.

The arithmetic lives in ``q8_oracle.c`` (plain C, fp64 where the pages do
not fix the precision); this module only builds it with gcc and marshals
numpy arrays through ctypes.  Every function is pinned by
``tests/test_oracle_pins.py``; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q8_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC", "-shared", "-std=c11"]

_lock = threading.Lock()
_lib = None

QK = 32
WBLK_BYTES = 34


def build(force: bool = False) -> str:
    """Compile q8_oracle.c with gcc into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_f32_to_f16.argtypes = [ctypes.c_float]
        lib.oracle_f32_to_f16.restype = ctypes.c_uint16
        lib.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f32.restype = ctypes.c_float
        lib.oracle_f32_to_f16_array.argtypes = [P, P, I64]
        lib.oracle_f16_to_f32_array.argtypes = [P, P, I64]
        lib.oracle_block_d32.argtypes = [P]
        lib.oracle_block_d32.restype = ctypes.c_float
        lib.oracle_quantize.argtypes = [P, I64, I64, P, P, I64]
        lib.oracle_rmsnorm.argtypes = [P, P, ctypes.c_float, I64, I64, P]
        lib.oracle_swiglu.argtypes = [P, P, I64, P]
        lib.oracle_gemm.argtypes = [P, I64, I64, P, P, P, I64, P, I64, P, P]
        lib.oracle_block_dots.argtypes = [P, I64, I64, P, I64, P]
        lib.oracle_q4a_gemm.argtypes = [P, I64, I64, P, P, P, I64, P, I64, P, P]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_div_reading_diff.argtypes = [P, I64, I64]
        lib.oracle_div_reading_diff.restype = ctypes.c_int64
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    """OpenMP threads the oracle uses (the cores it actually runs on)."""
    return int(_load().oracle_num_threads())


def f32_to_f16_bits(x) -> np.ndarray:
    """binary32 -> binary16 bits, round to nearest even (hand-written)."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_f32_to_f16_array(_ptr(x), _ptr(out), x.size)
    return out


def f16_bits_to_f32(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    _load().oracle_f16_to_f32_array(_ptr(h), _ptr(out), h.size)
    return out


def block_d32(block) -> float:
    """The f32 scale d = amax/127 of one 32-element block (before f16 storage)."""
    b = _c(block, np.float32)
    assert b.size == QK
    return float(_load().oracle_block_d32(_ptr(b)))


def quantize(x, rows_pad: int | None = None):
    """q8_0 plane of f32 rows x[rows][k]: (qs int8 [rows_pad][k], ds uint32 [rows_pad][k/32])."""
    x = _c(x, np.float32)
    rows, k = x.shape
    assert k % QK == 0
    rows_pad = rows if rows_pad is None else int(rows_pad)
    assert rows_pad >= rows
    qs = np.empty((rows_pad, k), dtype=np.int8)
    ds = np.empty((rows_pad, k // QK), dtype=np.uint32)
    _load().oracle_quantize(_ptr(x), rows, k, _ptr(qs), _ptr(ds), rows_pad)
    return qs, ds


def div_reading_diff(x) -> int:
    """Diagnostic: elements of f32 rows x[rows][k] whose q8_0 code would differ if
    the quantize step were read as rint(x/d) instead of the adopted rint(x*(1/d))."""
    x = _c(x, np.float32)
    rows, k = x.shape
    assert k % QK == 0
    return int(_load().oracle_div_reading_diff(_ptr(x), rows, k))


def unpack_ds(ds):
    """Split ds words into (f16 bits of d, int16 ssum)."""
    ds = np.asarray(ds, dtype=np.uint32)
    return (ds & 0xFFFF).astype(np.uint16), (ds >> 16).astype(np.uint16).view(np.int16)


def rmsnorm(x, w, eps: float):
    """fp64 y = (x * 1/sqrt(mean(x^2) + eps)) * w, per row."""
    x = _c(x, np.float32)
    w = _c(w, np.float32)
    rows, d = x.shape
    assert w.shape == (d,)
    y = np.empty((rows, d), dtype=np.float64)
    _load().oracle_rmsnorm(_ptr(x), _ptr(w), ctypes.c_float(eps), rows, d, _ptr(y))
    return y


def swiglu(g, u):
    """fp64 y = g / (1 + exp(-g)) * u, elementwise."""
    g = _c(g, np.float32)
    u = _c(u, np.float32)
    assert g.shape == u.shape
    y = np.empty(g.shape, dtype=np.float64)
    _load().oracle_swiglu(_ptr(g), _ptr(u), g.size, _ptr(y))
    return y


def gemm(w_blob, n: int, k: int, qs, ds, t_idx=None, n_idx=None):
    """fp64 y[t][n] = sum_b d_w * d_a * isum_b and absum = sum_b |term_b|.

    ``w_blob`` holds n rows of k/32 34-byte Q8_0 blocks; (qs, ds) is a plane
    with at least max(t_idx)+1 rows.  ``t_idx``/``n_idx`` select the
    sampled tokens/rows (default: all rows of the plane / all weight rows).
    """
    w_blob = _c(w_blob, np.uint8)
    qs = _c(qs, np.int8)
    ds = _c(ds, np.uint32)
    assert k % QK == 0 and w_blob.size == n * (k // QK) * WBLK_BYTES
    assert qs.shape[1] == k and ds.shape[1] == k // QK
    t_idx = np.arange(qs.shape[0], dtype=np.int64) if t_idx is None else _c(t_idx, np.int64)
    n_idx = np.arange(n, dtype=np.int64) if n_idx is None else _c(n_idx, np.int64)
    assert t_idx.size == 0 or (t_idx.min() >= 0 and t_idx.max() < qs.shape[0])
    assert n_idx.size == 0 or (n_idx.min() >= 0 and n_idx.max() < n)
    y = np.empty((t_idx.size, n_idx.size), dtype=np.float64)
    a = np.empty((t_idx.size, n_idx.size), dtype=np.float64)
    _load().oracle_gemm(_ptr(w_blob), n, k, _ptr(qs), _ptr(ds), _ptr(t_idx), t_idx.size,
                        _ptr(n_idx), n_idx.size, _ptr(y), _ptr(a))
    return y, a


Q4A_BLK_BYTES = 20  # f16 d, f16 m, 16 bytes of nibbles


def q4a_gemm(w_blob, n: int, k: int, qs, ds, t_idx=None, n_idx=None):
    """fp64 y[t][n] for asymmetric 4-bit weight blocks (value d*nib - m) and
    absum = sum_b (|d*d_a*isum_b| + |m*d_a*ssum_b|).

    ``w_blob`` holds n rows of k/32 20-byte blocks; the rest as in :func:`gemm`.
    """
    w_blob = _c(w_blob, np.uint8)
    qs = _c(qs, np.int8)
    ds = _c(ds, np.uint32)
    assert k % QK == 0 and w_blob.size == n * (k // QK) * Q4A_BLK_BYTES
    assert qs.shape[1] == k and ds.shape[1] == k // QK
    t_idx = np.arange(qs.shape[0], dtype=np.int64) if t_idx is None else _c(t_idx, np.int64)
    n_idx = np.arange(n, dtype=np.int64) if n_idx is None else _c(n_idx, np.int64)
    assert t_idx.size == 0 or (t_idx.min() >= 0 and t_idx.max() < qs.shape[0])
    assert n_idx.size == 0 or (n_idx.min() >= 0 and n_idx.max() < n)
    y = np.empty((t_idx.size, n_idx.size), dtype=np.float64)
    a = np.empty((t_idx.size, n_idx.size), dtype=np.float64)
    _load().oracle_q4a_gemm(_ptr(w_blob), n, k, _ptr(qs), _ptr(ds), _ptr(t_idx), t_idx.size,
                            _ptr(n_idx), n_idx.size, _ptr(y), _ptr(a))
    return y, a


def q4a_gemv(w_blob, n: int, k: int, qs, ds, n_idx=None):
    """Batch-1 form of :func:`q4a_gemm` (plane row 0): returns (y[n], absum[n])."""
    y, a = q4a_gemm(w_blob, n, k, qs, ds, t_idx=np.zeros(1, np.int64), n_idx=n_idx)
    return y[0], a[0]


def gemv(w_blob, n: int, k: int, qs, ds, n_idx=None):
    """Batch-1 case of :func:`gemm` on plane row 0: (y[n], absum[n])."""
    y, a = gemm(w_blob, n, k, qs, ds, t_idx=np.zeros(1, np.int64), n_idx=n_idx)
    return y[0], a[0]


def block_dots(w_blob, n: int, k: int, qs, t: int):
    """int32 isum[t][n][k/32] for tiny shapes."""
    w_blob = _c(w_blob, np.uint8)
    qs = _c(qs, np.int8)
    out = np.empty((t, n, k // QK), dtype=np.int32)
    _load().oracle_block_dots(_ptr(w_blob), n, k, _ptr(qs), t, _ptr(out))
    return out
