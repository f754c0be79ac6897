"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module draws random numbers and lays bytes out in the Q8_0 weight format.
It holds none of the method's arithmetic (no quantization, normalisation or
contraction), so both the CUDA path and the oracle can consume what it makes.

Recipes follow the workloads on the pages (all synthetic; no dataset):
  * Q8_0 weights: per-block f16 scale ~U(lo, hi) drawn in f32 and rounded to
    f16 by numpy, 32 int8 values ~U{-127..127}; each block is 34 bytes, the
    f16 scale (little-endian) then the 32 int8 values
    ("Part 4 - Lecture 05 - Fusion and the Activation-Quantization
    Discipline", sec. 2.1).
  * activations: f32 ~N(0, sigma) with an optional fraction of outliers
    multiplied by a constant.
Seeds are ``SeedSequence([config, tensor_id, ...])``.
"""
from __future__ import annotations

import numpy as np

QK = 32
WBLK_BYTES = 34


def rng(*key: int) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(k) for k in key]))


def pack_q8_0(d16_bits: np.ndarray, q: np.ndarray) -> np.ndarray:
    """Lay out (f16 bits [n][nb], int8 [n][nb*32]) as n rows of nb 34-byte blocks."""
    n, nb = d16_bits.shape
    assert q.shape == (n, nb * QK)
    out = np.empty((n, nb, WBLK_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = np.ascontiguousarray(d16_bits.astype("<u2")).view(np.uint8).reshape(n, nb, 2)
    out[:, :, 2:] = np.ascontiguousarray(q.astype(np.int8)).view(np.uint8).reshape(n, nb, QK)
    return out.reshape(-1)


def unpack_q8_0(blob: np.ndarray, n: int, k: int):
    """Inverse of :func:`pack_q8_0`: (f16 bits [n][nb], int8 [n][k])."""
    nb = k // QK
    b = np.asarray(blob, dtype=np.uint8).reshape(n, nb, WBLK_BYTES)
    d16 = np.ascontiguousarray(b[:, :, 0:2]).view("<u2").reshape(n, nb)
    q = np.ascontiguousarray(b[:, :, 2:]).view(np.int8).reshape(n, k)
    return d16.astype(np.uint16), q


def q8_0_weights(g: np.random.Generator, n: int, k: int, scale_lo: float = 0.002,
                 scale_hi: float = 0.02):
    """Random Q8_0 weight matrix: (blob uint8 [n*k/32*34], f16 bits [n][k/32], int8 [n][k])."""
    assert k % QK == 0
    nb = k // QK
    d = g.uniform(scale_lo, scale_hi, size=(n, nb)).astype(np.float32)
    d16 = d.astype(np.float16).view(np.uint16)
    q = g.integers(-127, 128, size=(n, k), dtype=np.int64).astype(np.int8)
    return pack_q8_0(d16, q), d16, q


Q4A_BLK_BYTES = 20  # asymmetric 4-bit block: f16 d, f16 m, 16 bytes of nibbles


def pack_q4a(d16_bits: np.ndarray, m16_bits: np.ndarray, nib: np.ndarray) -> np.ndarray:
    """Lay out (f16 d bits [n][nb], f16 m bits [n][nb], nibbles 0..15 [n][nb*32]) as n rows
    of nb 20-byte asymmetric blocks: d at +0, m at +2, then byte j (j < 16) holds element
    j in its low nibble and element j + 16 in its high nibble."""
    n, nb = d16_bits.shape
    assert m16_bits.shape == (n, nb) and nib.shape == (n, nb * QK)
    v = np.asarray(nib, dtype=np.uint8).reshape(n, nb, QK)
    assert int(v.max(initial=0)) <= 15
    out = np.empty((n, nb, Q4A_BLK_BYTES), dtype=np.uint8)
    out[:, :, 0:2] = np.ascontiguousarray(d16_bits.astype("<u2")).view(np.uint8).reshape(n, nb, 2)
    out[:, :, 2:4] = np.ascontiguousarray(m16_bits.astype("<u2")).view(np.uint8).reshape(n, nb, 2)
    out[:, :, 4:] = v[:, :, :16] | (v[:, :, 16:] << 4)
    return out.reshape(-1)


def q4a_weights(g: np.random.Generator, n: int, k: int, scale_lo: float = 0.001, scale_hi: float = 0.01):
    """Random asymmetric 4-bit weight matrix: (blob, f16 d bits, f16 m bits, nibbles [n][k]).

    d ~ U(scale_lo, scale_hi); m = d * U(0, 15) so that a block's values d*nib - m span
    an interval around zero (as an asymmetric min/max fit of roughly centred weights
    does); nibbles uniform in 0..15."""
    assert k % QK == 0
    nb = k // QK
    d = g.uniform(scale_lo, scale_hi, size=(n, nb)).astype(np.float32)
    m = (d * g.uniform(0.0, 15.0, size=(n, nb))).astype(np.float32)
    d16 = d.astype(np.float16).view(np.uint16)
    m16 = m.astype(np.float16).view(np.uint16)
    nib = g.integers(0, 16, size=(n, k), dtype=np.int64).astype(np.uint8)
    return pack_q4a(d16, m16, nib), d16, m16, nib


def activations(g: np.random.Generator, rows: int, k: int, sigma: float = 1.0,
                outlier_frac: float = 0.0, outlier_mult: float = 20.0) -> np.ndarray:
    """f32 ~N(0, sigma) [rows][k]; ``outlier_frac`` of the elements multiplied by ``outlier_mult``."""
    x = g.standard_normal(size=(rows, k), dtype=np.float32) * np.float32(sigma)
    if outlier_frac > 0.0:
        m = g.random(size=(rows, k)) < outlier_frac
        x[m] *= np.float32(outlier_mult)
    return x


def uniform(g: np.random.Generator, shape, lo: float, hi: float) -> np.ndarray:
    return g.uniform(lo, hi, size=shape).astype(np.float32)


# The five workloads (shapes only; seeds are the config numbers).
CONFIGS = {
    0: dict(name="tiny Q8_0 GEMV b=1", shapes=[(256, 512)], sigma=1.0, outlier_frac=0.0),
    1: dict(name="decode GEMV sweep b=1", shapes=[(12288, 7168), (96, 7168), (512, 128)],
            sigma=1.5, outlier_frac=0.01),
    2: dict(name="shared-activation decode", hidden=7168, eps=1e-6,
            shapes=[(3072, 7168), (512, 7168), (512, 7168), (3072, 7168)]),
    3: dict(name="prefill chain qwen2-7B-shaped", tokens=3325, d=3584, nf=18944, eps=1e-6),
    4: dict(name="layer-stack sweep", layers=28, d=3584, nf=18944, lm_head=152064,
            tokens=[1, 16, 512, 2048, 3325]),
}
