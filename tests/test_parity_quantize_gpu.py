"""GPU parity of the three quantizing kernels against the oracle.

The plane must equal the oracle's encoding bit for bit: of the given x for
quantize_q8_0, and of the f32 output the kernel itself wrote for the fused
producers (quantization is a pure function of the f32 bits, "54 - r51 -
producer-fused A-quantize mode 1", sec. 2.3).  Planes are pre-poisoned so
an unwritten byte (notably in the zero tail) shows up (sec. 4 of the same
page).  Shapes include the page's verifier set: nt = 1/63/64/129/3354 at
d = 3584, d = 896 nt = 300, d = 640 nt = 100, and nf = 18944.  Every fused
shape also runs in mode 2 (no f32 output), whose plane must be the mode-1
plane byte for byte.
"""
import numpy as np
import pytest

import oracle
from int8_quantized_projection_gb300 import synthetic as syn

from ._parity import assert_plane_equal, assert_y_close, dev, host, nan_f32, poisoned_plane

pytestmark = pytest.mark.gpu


def _edge_rows(k):
    """Rows of special blocks: zeros, single non-zero, +-amax ties, tiny amax, huge outliers."""
    rows = np.zeros((6, k), np.float32)
    rows[1, 5] = -3.25
    rows[2, 0::2] = 2.0
    rows[2, 1::2] = -2.0
    g = syn.rng(50, k)
    rows[3] = syn.activations(g, 1, k)[0] * np.float32(2.0 ** -100)
    rows[4] = syn.activations(g, 1, k, sigma=1.5, outlier_frac=0.05, outlier_mult=1000.0)[0]
    rows[5] = -0.0
    return rows


@pytest.mark.parametrize("rows,k,rows_pad", [(1, 32, 1), (1, 7168, 1), (5, 96, 128), (63, 3584, 128),
                                             (64, 3584, 64), (129, 640, 256), (300, 896, 300), (3354, 3584, 3456),
                                             # more rows than SMs: row groups (k <= 4096) or the flat stream
                                             (3325, 3584, 3328), (500, 32, 512), (1000, 4096, 1024),
                                             (153, 96, 153), (300, 4128, 384), (0, 256, 1024)])
def test_quantize_q8_0_bit_exact(q8, rows, k, rows_pad):
    g = syn.rng(51, rows, k)
    x = syn.activations(g, rows, k, sigma=1.5, outlier_frac=0.01)
    if rows >= 6:
        x[:6] = _edge_rows(k)
    qs, ds = poisoned_plane(rows_pad, k)
    q8.quantize_q8_0(dev(x), qs, ds)
    q8.q8_check()
    qr, dr = oracle.quantize(x, rows_pad)
    assert_plane_equal(qs, ds, qr, dr, f"quantize {rows}x{k}")


# Block maxima around the edge of the normal f32 range.  d = amax/127 is
# subnormal below 127 * 2^-126 = 1.49e-36, and 1/d overflows to infinity
# below about 127 * 2^-128 = 3.7e-37: there the products x * (1/d) are
# infinite and the clamp to +-127 decides every code, the one case where it
# can.  Every element is non-zero (0 * inf has no code).  Above 1.49e-36 d is
# normal and the clamp never changes a code.
TINY_AMAX = (1e-44, 1e-40, 1e-38, 1e-37, 3.6e-37, 3.8e-37, 1e-36, 1.4e-36, 1.6e-36, 1e-30)


def _tiny_rows(rows, k, seed):
    g = syn.rng(53, seed, rows, k)
    nb = k // 32
    mag = g.uniform(0.25, 1.0, size=(rows, k)).astype(np.float32)
    sign = np.where(g.integers(0, 2, size=(rows, k)) == 0, -1.0, 1.0).astype(np.float32)
    scale = np.array([TINY_AMAX[(r * nb + b) % len(TINY_AMAX)] for r in range(rows) for b in range(nb)],
                     np.float32).reshape(rows, nb)
    x = (sign * mag).reshape(rows, nb, 32) * scale[:, :, None]
    x = x.astype(np.float32)
    x[x == 0] = np.float32(1e-45)  # the smallest subnormal: no element underflows to 0
    return x.reshape(rows, k)


@pytest.mark.parametrize("rows,k,rows_pad", [(3, 320, 3), (2, 8192, 2), (700, 320, 704), (400, 4096, 512),
                                             (300, 4128, 384)])
def test_quantize_q8_0_subnormal_scales(q8, rows, k, rows_pad):
    """Blocks whose d is subnormal (and whose 1/d may be infinite): the codes
    the clamp decides, on the one-row, row-group and flat kernels."""
    x = _tiny_rows(rows, k, 1)
    assert (x != 0).all()
    qs, ds = poisoned_plane(rows_pad, k)
    q8.quantize_q8_0(dev(x), qs, ds)
    q8.q8_check()
    qr, dr = oracle.quantize(x, rows_pad)
    assert (np.abs(qr[:rows].astype(np.int32)) == 127).any()  # the data reaches the clamped case
    assert_plane_equal(qs, ds, qr, dr, f"quantize subnormal scales {rows}x{k}")


@pytest.mark.parametrize("rows,d,rows_pad", [(1, 3584, 1), (400, 3584, 512), (3, 8192, 3)])
def test_rmsnorm_quant_subnormal_outputs(q8, rows, d, rows_pad):
    """A norm weight small enough that y (and every block's d) is subnormal:
    the plane is still the exact encoding of the kernel's own y."""
    g = syn.rng(54, rows, d)
    x = syn.activations(g, rows, d)
    x = np.where(np.abs(x) < 1e-3, np.copysign(np.float32(1e-3), x), x).astype(np.float32)  # no y underflows to 0
    w = (syn.uniform(g, d, 0.5, 1.5) * np.float32(1e-38)).astype(np.float32)
    y = nan_f32(rows, d)
    qs, ds = poisoned_plane(rows_pad, d)
    q8.rmsnorm_quant(dev(x), dev(w), 1e-6, y, qs, ds)
    q8.q8_check()
    yh = host(y)
    assert (yh != 0).all() and np.abs(yh).max() < 1.49e-36  # no zero output; every block's d is subnormal
    qr, dr = oracle.quantize(yh, rows_pad)
    assert_plane_equal(qs, ds, qr, dr, f"rmsnorm subnormal plane {rows}x{d}")


def _tie_set(amax, g):
    """31 values below amax whose products with the block's 1/d round, in
    f32, to exactly k + 0.5 while the exact product is not k + 0.5: the code
    is rint of the rounded product (ties to even), and a kernel that formed
    the product and its rounding as one fused operation would get the other
    neighbour for about half of them."""
    d = np.float32(np.float32(amax) / np.float32(127))
    di = np.float32(np.float32(1) / d)
    out = []
    for k in g.permutation(np.arange(-126, 126)):
        v0 = np.float32((k + 0.5) / float(di))
        up = dn = v0
        cand = [v0]
        for _ in range(40):
            up = np.nextafter(up, np.float32(np.inf))
            dn = np.nextafter(dn, np.float32(-np.inf))
            cand += [up, dn]
        for v in cand:
            if (float(np.float32(v * di)) == k + 0.5 and float(v) * float(di) != k + 0.5
                    and abs(float(v)) < amax):
                out.append(v)
                break
        if len(out) == 31:
            return np.array(out, np.float32)
    raise AssertionError("too few tie values")


def _tie_rows(rows, k):
    g = syn.rng(55, rows, k)
    amaxes = (1.0, 3.7, 0.013, 250.0, 0.5, 17.25)
    sets = [_tie_set(a, g) for a in amaxes]
    nb = rows * k // 32
    pick = g.integers(0, len(amaxes), size=nb)
    blocks = np.empty((nb, 32), np.float32)
    for j, a in enumerate(amaxes):
        sel = np.flatnonzero(pick == j)
        vals = np.concatenate([np.full((len(sel), 1), a, np.float32), np.tile(sets[j], (len(sel), 1))], axis=1)
        vals *= np.where(g.integers(0, 2, size=vals.shape) == 0, -1.0, 1.0).astype(np.float32)
        blocks[sel] = np.take_along_axis(vals, g.permuted(np.tile(np.arange(32), (len(sel), 1)), axis=1), axis=1)
    return blocks.reshape(rows, k)


@pytest.mark.parametrize("rows,k,rows_pad", [(2, 640, 2), (300, 640, 384), (3325, 3584, 3328), (200, 8192, 256)])
def test_quantize_q8_0_product_ties(q8, rows, k, rows_pad):
    """Every block holds its amax and 31 elements whose f32 product with 1/d
    lands exactly on k + 0.5 ("54 - r51 - producer-fused A-quantize mode 1",
    sec. 3.2: the code is rint of x times the f32 reciprocal of d, ties to
    even), on the one-row, row-group and flat kernels."""
    x = _tie_rows(rows, k)
    b = x.reshape(-1, 32)
    d = (np.abs(b).max(axis=1) / np.float32(127)).astype(np.float32)
    di = (np.float32(1) / d).astype(np.float32)
    p = (b * di[:, None]).astype(np.float32)
    split = np.rint(p) != np.rint(b.astype(np.float64) * di[:, None].astype(np.float64))
    assert split.sum() > len(b)  # the data reaches the case, more than once per block on average
    qs, ds = poisoned_plane(rows_pad, k)
    q8.quantize_q8_0(dev(x), qs, ds)
    q8.q8_check()
    qr, dr = oracle.quantize(x, rows_pad)
    assert_plane_equal(qs, ds, qr, dr, f"quantize product ties {rows}x{k}")


def test_quantize_q8_0_zero_rows_only_fills_tail(q8):
    import torch

    qs, ds = poisoned_plane(128, 64)
    q8.quantize_q8_0(torch.empty((0, 64), dtype=torch.float32, device="cuda"), qs, ds)
    q8.q8_check()
    assert (host(qs) == 0).all() and (host(ds) == 0).all()


@pytest.mark.parametrize("rows,d,rows_pad", [(1, 3584, 1), (63, 3584, 64), (64, 3584, 64), (129, 3584, 192),
                                             (300, 896, 384), (100, 640, 128), (1, 7168, 1), (7, 18944, 8),
                                             (3354, 3584, 3456), (2, 32768, 2),
                                             (3, 8192, 3), (3, 8224, 4),  # weight vector staged / read directly
                                             # more rows than SMs: the shared-memory row ring (up to d = 16384)
                                             (3325, 3584, 3328), (1000, 8192, 1024), (500, 32, 512),
                                             (400, 16384, 512), (153, 896, 153), (300, 16416, 384)])
def test_rmsnorm_quant(q8, rows, d, rows_pad):
    import torch

    g = syn.rng(52, rows, d)
    x = syn.activations(g, rows, d)
    if rows >= 6:
        x[:6] = _edge_rows(d)
        x[0, 0] = 1.0  # avoid an all-zero row (ss = 0 -> finite scale, but a degenerate case covered below)
    w = syn.uniform(g, d, 0.5, 1.5)
    eps = 1e-6
    y = nan_f32(rows, d)
    qs, ds = poisoned_plane(rows_pad, d)
    q8.rmsnorm_quant(dev(x), dev(w), eps, y, qs, ds)
    q8.q8_check()
    assert_y_close(y, oracle.rmsnorm(x, w, eps), f"rmsnorm y {rows}x{d}")
    qr, dr = oracle.quantize(host(y), rows_pad)
    assert_plane_equal(qs, ds, qr, dr, f"rmsnorm plane {rows}x{d}")
    # fused == the standalone quantizer applied to the kernel's own output
    qs2, ds2 = poisoned_plane(rows_pad, d)
    q8.quantize_q8_0(y, qs2, ds2)
    q8.q8_check()
    assert torch.equal(qs, qs2) and torch.equal(ds, ds2)
    # mode 2 (no f32 output): the same plane, byte for byte
    qs3, ds3 = poisoned_plane(rows_pad, d)
    q8.rmsnorm_quant(dev(x), dev(w), eps, None, qs3, ds3)
    q8.q8_check()
    assert torch.equal(qs, qs3) and torch.equal(ds, ds3)


def test_rmsnorm_quant_zero_row(q8):
    x = np.zeros((2, 256), np.float32)
    x[1] = 1.0
    w = np.ones(256, np.float32)
    y = nan_f32(2, 256)
    qs, ds = poisoned_plane(2, 256)
    q8.rmsnorm_quant(dev(x), dev(w), 1e-6, y, qs, ds)
    q8.q8_check()
    assert_y_close(y, oracle.rmsnorm(x, w, 1e-6), "zero row")
    assert (host(qs)[0] == 0).all() and (host(ds)[0] == 0).all()


@pytest.mark.parametrize("rows,nf,rows_pad", [(1, 18944, 1), (63, 18944, 64), (65, 4096, 128),
                                              (100, 640, 128), (3325, 18944, 3328)])
def test_swiglu_quant(q8, rows, nf, rows_pad):
    import torch

    g = syn.rng(53, rows, nf)
    gate = syn.activations(g, rows, nf)
    up = syn.activations(g, rows, nf)
    if rows >= 2:
        gate[0, :64] = np.array([-100.0, -88.0, -80.0, 0.0, 30.0, 90.0] * 10 + [1, 2, 3, 4], np.float32)
        up[1] = 0.0
    y = nan_f32(rows, nf)
    qs, ds = poisoned_plane(rows_pad, nf)
    q8.swiglu_quant(dev(gate), dev(up), y, qs, ds)
    q8.q8_check()
    assert_y_close(y, oracle.swiglu(gate, up), f"swiglu y {rows}x{nf}")
    qr, dr = oracle.quantize(host(y), rows_pad)
    assert_plane_equal(qs, ds, qr, dr, f"swiglu plane {rows}x{nf}")
    qs2, ds2 = poisoned_plane(rows_pad, nf)
    q8.quantize_q8_0(y, qs2, ds2)
    q8.q8_check()
    assert torch.equal(qs, qs2) and torch.equal(ds, ds2)
    # mode 2 (no f32 output): the same plane, byte for byte
    qs3, ds3 = poisoned_plane(rows_pad, nf)
    q8.swiglu_quant(dev(gate), dev(up), None, qs3, ds3)
    q8.q8_check()
    assert torch.equal(qs, qs3) and torch.equal(ds, ds3)


def test_quantizers_are_deterministic(q8):
    import torch

    g = syn.rng(54, 0)
    x = dev(syn.activations(g, 257, 3584))
    w = dev(syn.uniform(g, 3584, 0.5, 1.5))
    outs = []
    for _ in range(2):
        y = nan_f32(257, 3584)
        qs, ds = poisoned_plane(384, 3584)
        q8.rmsnorm_quant(x, w, 1e-6, y, qs, ds)
        q8.q8_check()
        outs.append((y.view(torch.int32).clone(), qs.clone(), ds.clone()))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
