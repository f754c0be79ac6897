"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test compares the oracle with something independent of its code: numpy's
own float16 conversion, Python's half-to-even ``round``, exact rational
arithmetic (``fractions``), closed forms, Python-int brute force, numpy's
int64 matmul, and the byte accounts printed on the pages.  A plausible slip
anywhere in the oracle (a wrong constant, a dropped term, a transposed
operand, a wrong sign, a wrong packing) fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from int8_quantized_projection_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# f32 <-> f16 (IEEE 754): against numpy's conversion
# --------------------------------------------------------------------------

def _check_f16_chunk(bits_u32):
    f = bits_u32.view(np.float32)
    mine = oracle.f32_to_f16_bits(f)
    ref = f.astype(np.float16).view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.all((mine[nan] & 0x7C00) == 0x7C00) and np.all((mine[nan] & 0x3FF) != 0)


def test_f32_to_f16_exhaustive_over_the_rounding_range():
    # Every f32 whose exponent byte lies in [96, 143] (|x| in [2^-31, 2^17)),
    # both signs: all of them round to something other than a trivial 0/inf.
    with np.errstate(over="ignore"):
        for sign in (0, 1):
            for eb in range(96, 144):
                base = (sign << 31) | (eb << 23)
                _check_f16_chunk(np.arange(base, base + (1 << 23), dtype=np.uint32))


def test_f32_to_f16_outside_the_rounding_range():
    g = syn.rng(99, 0)
    with np.errstate(over="ignore"):
        for sign in (0, 1):
            for eb in list(range(0, 96)) + list(range(144, 256)):
                base = (sign << 31) | (eb << 23)
                m = g.integers(0, 1 << 23, size=4096, dtype=np.uint32)
                m[:2] = [0, (1 << 23) - 1]
                _check_f16_chunk((np.uint32(base) | m).astype(np.uint32))


def test_f16_to_f32_exhaustive():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    mine = oracle.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(mine[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    assert np.all(np.isnan(mine[nan]))


# --------------------------------------------------------------------------
# q8_0 quantization ("54 - r51 - producer-fused A-quantize mode 1", sec. 2.1, 3.2)
# --------------------------------------------------------------------------

def _quant_block(x):
    qs, ds = oracle.quantize(np.asarray(x, np.float32).reshape(1, 32))
    d16, ssum = oracle.unpack_ds(ds)
    return qs[0], int(d16[0, 0]), int(ssum[0, 0])


def test_quantize_ties_round_half_to_even():
    # amax = 127 gives d = 1 and di = 1, so x*di = x exactly and every
    # x = k + 0.5 is a tie; Python's round() is half-to-even.
    for k in range(-127, 127, 31):
        vals = [127.0] + [k + 0.5 + j for j in range(31) if -127 < k + 0.5 + j < 127][:31]
        vals += [0.0] * (32 - len(vals))
        q, d16, ssum = _quant_block(vals)
        expect = [round(v) for v in vals]
        assert list(q) == expect
        assert ssum == sum(expect)
        assert d16 == 0x3C00  # f16 1.0


@pytest.mark.parametrize("e", [-20, -7, -1, 0, 3, 9])
def test_quantize_power_of_two_scale_exact(e):
    # amax = 127 * 2^e gives d = 2^e and di = 2^-e exactly, so the codes are
    # round_half_even(x / 2^e) computed exactly with fractions.
    g = syn.rng(98, e + 100)
    x = (g.uniform(-127, 127, 32) * 2.0 ** e).astype(np.float32)
    x[5] = np.float32(-127 * 2.0 ** e)
    q, d16, ssum = _quant_block(x)
    expect = [round(Fraction(float(v)) / Fraction(2) ** e) for v in x]
    assert list(q) == expect
    assert ssum == sum(expect)
    assert d16 == int(np.float16(2.0 ** e).view(np.uint16))


def _blocks_for_round_trip():
    g = syn.rng(97, 1)
    out = [syn.activations(g, 64, 32, sigma=1.0)]
    out.append(syn.activations(g, 64, 32, sigma=1.5, outlier_frac=0.05))
    out.append((syn.activations(g, 16, 32) * np.float32(2.0 ** -100)).astype(np.float32))
    out.append((syn.activations(g, 16, 32) * np.float32(1000.0)).astype(np.float32))
    z = np.zeros((4, 32), np.float32)
    z[1, 7] = 3.5            # single non-zero
    z[2, :] = -0.0           # all negative zero
    z[3, ::2] = 2.0
    z[3, 1::2] = -2.0        # +-amax ties
    out.append(z)
    return np.concatenate(out)


def test_quantize_round_trip_and_invariants():
    x = _blocks_for_round_trip()
    qs, ds = oracle.quantize(x)
    d16, ssum = oracle.unpack_ds(ds)
    for i in range(x.shape[0]):
        xb = x[i].astype(np.float64)
        q = qs[i].astype(np.int64)
        amax = float(np.max(np.abs(xb)))
        d32 = oracle.block_d32(x[i])
        # d is amax/127 up to one f32 rounding
        assert abs(d32 * 127.0 - amax) <= amax * 2.0 ** -23
        # the stored scale is d rounded to f16 (numpy's conversion)
        assert int(d16[i, 0]) == int(np.float32(d32).astype(np.float16).view(np.uint16))
        # round trip |x - q*d| <= d/2, plus the slack of two f32 roundings in x*di
        assert np.all(np.abs(xb - q * d32) <= d32 * (0.5 + 2.0 ** -15))
        # ssum invariant and range
        assert int(ssum[i, 0]) == int(q.sum()) and abs(int(ssum[i, 0])) <= 32 * 127
        assert q.min() >= -127 and q.max() <= 127
        if amax > 0:
            j = int(np.argmax(np.abs(xb)))
            assert abs(int(q[j])) == 127 and np.sign(q[j]) == np.sign(xb[j])
        else:
            assert np.all(q == 0) and int(ds[i, 0]) == 0


def test_quantize_plane_layout_and_zero_tail():
    g = syn.rng(97, 2)
    x = syn.activations(g, 5, 96)
    qs, ds = oracle.quantize(x, rows_pad=8)
    assert qs.shape == (8, 96) and ds.shape == (8, 3)
    assert np.all(qs[5:] == 0) and np.all(ds[5:] == 0)
    # rows and blocks are independent: quantizing one block alone gives the same bytes
    q1, d1 = oracle.quantize(x[3:4, 32:64])
    assert np.array_equal(q1[0], qs[3, 32:64]) and int(d1[0, 0]) == int(ds[3, 1])
    # ds packs d (bits 0..15) and ssum (bits 16..31)
    d16, ssum = oracle.unpack_ds(ds[:5])
    assert np.array_equal(ssum.astype(np.int64), qs[:5].reshape(5, 3, 32).astype(np.int64).sum(-1))
    assert np.all(d16 != 0)


# --------------------------------------------------------------------------
# RMSNorm and SwiGLU ("54 - r51 - producer-fused A-quantize mode 1", sec. 3.2)
# --------------------------------------------------------------------------

def test_rmsnorm_constant_row_closed_form():
    # x = c everywhere: mean(x^2) = c^2, so y_i = c * w_i / sqrt(c^2 + eps).
    g = syn.rng(96, 1)
    d = 640
    w = syn.uniform(g, d, 0.5, 1.5)
    for c, eps in [(0.75, 1e-6), (-3.0, 1e-6), (1e-3, 1e-6), (2.5, 0.5)]:
        x = np.full((1, d), c, np.float32)
        y = oracle.rmsnorm(x, w, eps)[0]
        cc = float(np.float32(c))
        ref = cc * w.astype(np.float64) / math.sqrt(cc * cc + float(np.float32(eps)))
        assert np.allclose(y, ref, rtol=1e-12, atol=0)


def test_rmsnorm_unit_rms_invariant():
    # With w = 1 and eps = 0 the output has mean square exactly 1 and is
    # proportional to x (positive factor).
    g = syn.rng(96, 2)
    x = syn.activations(g, 4, 3584, sigma=2.0)
    y = oracle.rmsnorm(x, np.ones(3584, np.float32), 0.0)
    assert np.allclose((y * y).mean(axis=1), 1.0, rtol=1e-12)
    ratio = y / x.astype(np.float64)
    assert np.all(ratio > 0) and np.allclose(ratio, ratio[:, :1], rtol=1e-12)


def test_swiglu_closed_forms():
    u = np.array([1.0, -2.5, 3.0, 0.5], np.float32)
    y = oracle.swiglu(np.zeros(4, np.float32), u)
    assert np.all(y == 0.0)
    l3 = np.float32(math.log(3.0))
    y = oracle.swiglu(np.full(4, l3, np.float32), u)          # sigmoid(ln 3) = 3/4
    # f32(ln 3) is ln 3 to within 2^-24 relative, which moves sigmoid by < 2e-8
    assert np.allclose(y, 0.75 * float(l3) * u.astype(np.float64), rtol=1e-7)
    y = oracle.swiglu(np.full(4, 40.0, np.float32), u)         # g large: y -> g*u
    assert np.allclose(y, 40.0 * u.astype(np.float64), rtol=1e-15)


def test_swiglu_odd_part_identity():
    # silu(g) - silu(-g) = g, so y(g, u) - y(-g, u) = g * u.
    g = syn.rng(96, 3)
    gv = syn.activations(g, 1, 4096)[0]
    uv = syn.activations(g, 1, 4096)[0]
    lhs = oracle.swiglu(gv, uv) - oracle.swiglu(-gv, uv)
    rhs = gv.astype(np.float64) * uv.astype(np.float64)
    assert np.allclose(lhs, rhs, rtol=1e-13, atol=1e-300)


# --------------------------------------------------------------------------
# Q8_0 x q8_0 contraction ("Part 4 - Lecture 05", sec. 2.1-2.2)
# --------------------------------------------------------------------------

def _brute_block_dots(blob, n, k, qs, t):
    raw = bytes(np.asarray(blob, np.uint8))
    nb = k // 32
    out = np.zeros((t, n, nb), dtype=np.int64)
    for i in range(t):
        arow = [int(v) for v in qs[i]]
        for j in range(n):
            for b in range(nb):
                off = (j * nb + b) * 34 + 2
                wq = [v - 256 if v > 127 else v for v in raw[off:off + 32]]
                out[i, j, b] = sum(a * c for a, c in zip(wq, arow[b * 32:(b + 1) * 32]))
    return out


def test_block_dots_bruteforce_python_ints():
    g = syn.rng(95, 1)
    for n, k, t in [(3, 64, 2), (8, 256, 3), (5, 96, 1)]:
        blob, _, q = syn.q8_0_weights(g, n, k)
        qa = g.integers(-127, 128, size=(t, k)).astype(np.int8)
        if n >= 3:
            # extreme patterns: all +127 against +-127, and +127 against -127
            bq = blob.reshape(n, k // 32, 34)
            bq[0, :, 2:] = np.uint8(127)
            bq[1, :, 2:] = np.int8(-127).view(np.uint8)
            qa[0, :] = 127
        got = oracle.block_dots(blob, n, k, qa, t)
        assert np.array_equal(got.astype(np.int64), _brute_block_dots(blob, n, k, qa, t))
    assert _brute_block_dots(blob, n, k, qa, t).__abs__().max() <= 32 * 127 * 127


def _plane_from(qa, d16_bits):
    qa = np.asarray(qa, np.int8)
    t, k = qa.shape
    ssum = qa.reshape(t, k // 32, 32).astype(np.int64).sum(-1)
    ds = (d16_bits.astype(np.uint32) | ((ssum.astype(np.int16).view(np.uint16).astype(np.uint32)) << 16))
    return qa, ds.astype(np.uint32)


def test_gemm_all_scales_one_is_integer_matmul():
    g = syn.rng(95, 2)
    n, k, t = 24, 512, 7
    _, _, q = syn.q8_0_weights(g, n, k)
    blob = syn.pack_q8_0(np.full((n, k // 32), 0x3C00, np.uint16), q)
    qa = g.integers(-127, 128, size=(t, k)).astype(np.int8)
    qs, ds = _plane_from(qa, np.full((t, k // 32), 0x3C00, np.uint16))
    y, a = oracle.gemm(blob, n, k, qs, ds)
    ref = qa.astype(np.int64) @ q.astype(np.int64).T
    assert np.array_equal(y, ref.astype(np.float64))
    assert np.all(a >= np.abs(y))


def test_gemm_exact_rational_small():
    # Random f16 scales on both sides: the oracle's fp64 sum agrees with the
    # exact rational value within the rounding of a short fp64 sum.
    g = syn.rng(95, 3)
    n, k, t = 6, 192, 3
    blob, dw16, q = syn.q8_0_weights(g, n, k)
    qa = g.integers(-127, 128, size=(t, k)).astype(np.int8)
    da16 = g.uniform(1e-3, 5e-2, size=(t, k // 32)).astype(np.float16).view(np.uint16)
    qs, ds = _plane_from(qa, da16)
    y, a = oracle.gemm(blob, n, k, qs, ds)
    nb = k // 32
    for i in range(t):
        for j in range(n):
            exact = Fraction(0)
            for b in range(nb):
                isum = int(np.dot(q[j, b * 32:(b + 1) * 32].astype(np.int64), qa[i, b * 32:(b + 1) * 32].astype(np.int64)))
                exact += (Fraction(float(dw16[j, b:b + 1].view(np.float16)[0]))
                          * Fraction(float(da16[i, b:b + 1].view(np.float16)[0])) * isum)
            assert abs(Fraction(y[i, j]) - exact) <= Fraction(a[i, j]) * Fraction(1, 2 ** 48)


def test_gemm_sampling_matches_full():
    g = syn.rng(95, 4)
    n, k = 40, 256
    blob, _, _ = syn.q8_0_weights(g, n, k)
    qs, ds = oracle.quantize(syn.activations(g, 9, k))
    y, a = oracle.gemm(blob, n, k, qs, ds)
    ti, ni = np.array([8, 0, 3]), np.array([39, 2, 17, 5])
    ys, as_ = oracle.gemm(blob, n, k, qs, ds, t_idx=ti, n_idx=ni)
    assert np.array_equal(ys, y[np.ix_(ti, ni)]) and np.array_equal(as_, a[np.ix_(ti, ni)])
    yv, av = oracle.gemv(blob, n, k, qs, ds)
    assert np.array_equal(yv, y[0]) and np.array_equal(av, a[0])


def test_weight_layout_round_trip():
    g = syn.rng(95, 5)
    blob, d16, q = syn.q8_0_weights(g, 3, 64)
    d16b, qb = syn.unpack_q8_0(blob, 3, 64)
    assert np.array_equal(d16b, d16) and np.array_equal(qb, q)
    raw = blob.reshape(3, 2, 34)
    assert int(raw[1, 1, 0]) | (int(raw[1, 1, 1]) << 8) == int(d16[1, 1])  # little-endian f16 at +0
    assert np.array_equal(raw[2, 0, 2:].view(np.int8), q[2, :32])          # int8 qs at +2


# --------------------------------------------------------------------------
# Asymmetric 4-bit weight blocks (value d*nib - m) and the ssum min term
# --------------------------------------------------------------------------

def test_q4a_block_layout_literal():
    # d = 1.0 (f16 0x3C00), m = 2.0 (0x4000), element j = j % 16: byte j (j < 16)
    # holds element j in its low nibble and element j + 16 in its high nibble
    d16 = np.array([[0x3C00]], np.uint16)
    m16 = np.array([[0x4000]], np.uint16)
    nib = (np.arange(32) % 16).astype(np.uint8).reshape(1, 32)
    blob = syn.pack_q4a(d16, m16, nib)
    expect = bytes([0x00, 0x3C, 0x00, 0x40] + [0x11 * j for j in range(16)])
    assert blob.tobytes() == expect


def _q4a_exact(d16, m16, nib, qa, da16, i, j, k):
    """Exact rational sum over the elements of (d*nib - m) * (d_a*q), from the
    dequantized values themselves (no block sums, no ssum identity)."""
    h = lambda bits: Fraction(float(np.array([bits], np.uint16).view(np.float16)[0]))
    tot = Fraction(0)
    for e in range(k):
        b = e // 32
        wv = h(d16[j, b]) * int(nib[j, e]) - h(m16[j, b])
        tot += wv * h(da16[i, b]) * int(qa[i, e])
    return tot


def test_q4a_exact_rational_small():
    g = syn.rng(96, 1)
    n, k, t = 5, 160, 3
    blob, d16, m16, nib = syn.q4a_weights(g, n, k)
    qa = g.integers(-127, 128, size=(t, k)).astype(np.int8)
    qa[0, :32] = 0           # a zero activation block (ssum = 0)
    qa[1, 32:64] = -127      # a saturated one (ssum = -4064)
    da16 = g.uniform(1e-3, 5e-2, size=(t, k // 32)).astype(np.float16).view(np.uint16)
    qs, ds = _plane_from(qa, da16)
    y, a = oracle.q4a_gemm(blob, n, k, qs, ds)
    for i in range(t):
        for j in range(n):
            exact = _q4a_exact(d16, m16, nib, qa, da16, i, j, k)
            assert abs(Fraction(y[i, j]) - exact) <= Fraction(a[i, j]) * Fraction(1, 2 ** 48)


def test_q4a_zero_min_is_the_q8_0_contraction():
    # m = 0: the block is d*nib, i.e. a Q8_0 block with codes nib and the same d
    g = syn.rng(96, 2)
    n, k = 7, 256
    _, d16, _, nib = syn.q4a_weights(g, n, k)
    blob4 = syn.pack_q4a(d16, np.zeros_like(d16), nib)
    blob8 = syn.pack_q8_0(d16, nib.astype(np.int8))
    qs, ds = oracle.quantize(syn.activations(g, 4, k))
    y4, a4 = oracle.q4a_gemm(blob4, n, k, qs, ds)
    y8, a8 = oracle.gemm(blob8, n, k, qs, ds)
    assert np.array_equal(y4, y8) and np.array_equal(a4, a8)


def test_q4a_constant_weights_reduce_to_the_activation_sum():
    # nib = 0 everywhere: every weight is -m, so y = -m * sum_e xhat_e, a plain
    # sum of the dequantized activation (numpy fp64 over exact products)
    g = syn.rng(96, 3)
    n, k, t = 3, 128, 2
    d16 = np.full((n, k // 32), 0x2000, np.uint16)           # 2^-7
    m16 = np.array([[0x3800], [0x3C00], [0x4000]], np.uint16).repeat(k // 32, 1)  # 0.5, 1, 2
    blob = syn.pack_q4a(d16, m16, np.zeros((n, k), np.uint8))
    qs, ds = oracle.quantize(syn.activations(g, t, k))
    y, _ = oracle.q4a_gemm(blob, n, k, qs, ds)
    da = (ds & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)
    xhat = qs.astype(np.float64) * np.repeat(da, 32, axis=1)
    for j, mv in enumerate((0.5, 1.0, 2.0)):
        np.testing.assert_allclose(y[:, j], -mv * xhat.sum(axis=1), rtol=1e-13, atol=1e-13)


def test_q4a_sampling_and_gemv_match_full():
    g = syn.rng(96, 4)
    n, k = 30, 256
    blob, _, _, _ = syn.q4a_weights(g, n, k)
    qs, ds = oracle.quantize(syn.activations(g, 5, k))
    y, a = oracle.q4a_gemm(blob, n, k, qs, ds)
    ti, ni = np.array([4, 0]), np.array([29, 3, 11])
    ys, as_ = oracle.q4a_gemm(blob, n, k, qs, ds, t_idx=ti, n_idx=ni)
    assert np.array_equal(ys, y[np.ix_(ti, ni)]) and np.array_equal(as_, a[np.ix_(ti, ni)])
    yv, av = oracle.q4a_gemv(blob, n, k, qs, ds)
    assert np.array_equal(yv, y[0]) and np.array_equal(av, a[0])


# --------------------------------------------------------------------------
# Byte accounts printed on the pages (tests/golden/page_byte_accounts.json)
# --------------------------------------------------------------------------

def test_page_byte_accounts():
    with open(os.path.join(GOLDEN, "page_byte_accounts.json")) as f:
        entries = json.load(f)["entries"]
    for e in entries:
        if "n" in e:
            g = syn.rng(94, 0)
            blob, _, _ = syn.q8_0_weights(g, 2, e["k"])
            wbytes = blob.nbytes // 2 * e["n"]
            if e["printed"] == 94:
                got = wbytes
            else:  # each output row re-reads the ~28 KB f32 activation
                got = e["k"] * 4 * e["n"]
                assert abs(got / wbytes - e["ratio_printed"]) <= e["ratio_tol"]
        elif e["part"] == "f32":
            got = e["rows"] * e["k"] * np.dtype(np.float32).itemsize
        else:
            x = np.zeros((1, e["k"]), np.float32)
            qs, ds = oracle.quantize(x, rows_pad=e["rows_pad"])
            got = qs.nbytes if e["part"] == "qs" else ds.nbytes
            if "exact" in e:
                assert got == e["exact"]
        assert abs(got / 1e6 - e["printed"]) <= e["rel_tol"] * e["printed"], e["what"]


# --------------------------------------------------------------------------
# The x/d reading of the quantize step against the adopted x*(1/d) reading
# ("54 - r51 - producer-fused A-quantize mode 1", sec. 3.2 prints the product
# form; the plain definition is q = rint(x/d)).  A diagnostic count, pinned to
# numpy's IEEE f32 arithmetic, then reported on the workloads' activations.
# --------------------------------------------------------------------------

def _div_reading_diff_numpy(x):
    b = x.astype(np.float32).reshape(x.shape[0], -1, 32)
    d = (np.abs(b).max(-1, keepdims=True) / np.float32(127)).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        di = np.where(d != 0, np.float32(1) / d, np.float32(0)).astype(np.float32)
        q_mul = np.clip(np.rint((b * di).astype(np.float32)), -127, 127)
        q_div = np.where(d != 0, np.clip(np.rint((b / d).astype(np.float32)), -127, 127), 0)
    return int((q_mul != q_div).sum())


def test_div_reading_diagnostic_matches_numpy():
    g = syn.rng(95, 0)
    x = syn.activations(g, 2000, 4096, sigma=1.5, outlier_frac=0.01)
    got = oracle.div_reading_diff(x)
    assert got == _div_reading_diff_numpy(x)
    assert got > 0  # the two readings do differ on some of these 8 M elements
    # a constant block: x = amax, both readings give exactly 127
    assert oracle.div_reading_diff(np.full((1, 32), 3.0, np.float32)) == 0


def test_div_reading_count_on_the_workloads(capsys):
    """Elements whose code the other reading would change, per workload
    activation recipe.  The two forms differ only by an f32 rounding or two,
    so only values within a few ulp of a half-integer step can change: about
    one code in a million."""
    cases = {"decode x (1 x 7168, N(0,1.5), 1% x20)": syn.activations(syn.rng(1, 0), 1, 7168, 1.5, 0.01),
             "prefill x (3325 x 3584, N(0,1))": syn.activations(syn.rng(3, 0), 3325, 3584),
             "prefill SwiGLU width (3325 x 18944, N(0,1))": syn.activations(syn.rng(3, 9), 3325, 18944)}
    for name, x in cases.items():
        c = oracle.div_reading_diff(x)
        with capsys.disabled():
            print(f"\n  x/d vs x*(1/d): {c} of {x.size} codes differ on {name}")
        assert c <= 4e-6 * x.size
