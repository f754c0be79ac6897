"""GPU parity of q8_0_gemv_fused: the one-row producer computed inside the
GEMV's activation staging ("Part 4 - Lecture 05", sec. 4: producer and
consumer in one launch, one implementation for both paths).

Every output must equal, bit for bit, the two-launch path it replaces: the
standalone producer on one row (rows_pad = q8_plane_rows(1)) followed by
q8_0_gemv_grouped on its plane.  That path is itself pinned to the oracle
(the producers' planes bit-exact, the GEMV within its tolerance); here the
fused outputs are also compared with the oracle's GEMV of the oracle's
encoding of the producer's f32 row.  Shapes cover one and several
projections, CTAs with few warps (small n: the RMSNorm sum of squares is
then replayed by fewer warps than the standalone kernel has), rows of one
and of several 32-chunk pieces, and the largest k of each producer.
"""
import numpy as np
import pytest

import oracle
from int8_quantized_projection_gb300 import synthetic as syn

from ._parity import assert_gemm_close, dev, host, nan_f32

pytestmark = pytest.mark.gpu

CASES = [
    # (k, ns)
    (256, (64,)),
    (512, (256,)),      # the tiny configuration: 16 blocks per row, one launch per step
    (3584, (3584, 512, 512)),
    (3584, (37,)),
    (7168, (3072, 512, 512, 3072)),
    (7168, (96,)),
    (18944, (3584,)),
    (32768, (1000, 8)),
]


def _weights(seed, n, k):
    return syn.q8_0_weights(syn.rng(70, seed, n, k), n, k)[0]


def _inputs(producer, k, seed):
    g = syn.rng(71, seed, producer, k)
    a = syn.activations(g, 1, k, sigma=1.5, outlier_frac=0.01)[0]
    b = syn.activations(g, 1, k)[0] if producer == 3 else None
    w = syn.uniform(g, k, 0.5, 1.5) if producer == 2 else None
    return a, b, w


def _two_launch(q8, producer, k, a, b, w, eps, projs):
    """The standalone producer (mode 1, one row) and the grouped GEMV on its plane."""
    rp = q8.q8_plane_rows(1)
    qs, ds = q8.empty_plane(rp, k)
    yf = nan_f32(1, k)
    if producer == q8.PRODUCER_QUANT:
        q8.quantize_q8_0(a.view(1, k), qs, ds)
        yf = a.view(1, k)
    elif producer == q8.PRODUCER_RMSNORM:
        q8.rmsnorm_quant(a.view(1, k), w, eps, yf, qs, ds)
    else:
        q8.swiglu_quant(a.view(1, k), b.view(1, k), yf, qs, ds)
    q8.q8_0_gemv_grouped(projs, k, qs, ds)
    q8.q8_check()
    return yf


@pytest.mark.parametrize("producer", [1, 2, 3])
@pytest.mark.parametrize("k,ns", CASES)
def test_fused_equals_two_launches_and_oracle(q8, producer, k, ns):
    import torch

    if producer == 2 and k > 32768:
        pytest.skip("RMSNorm rows are limited to 32768")
    a_h, b_h, w_h = _inputs(producer, k, len(ns))
    a, b, w = dev(a_h), (dev(b_h) if b_h is not None else None), (dev(w_h) if w_h is not None else None)
    eps = 1e-6
    blobs = [_weights(i, n, k) for i, n in enumerate(ns)]
    wd = [dev(bl) for bl in blobs]
    yf_fused = [nan_f32(n) for n in ns]
    q8.q8_0_gemv_fused([(x, n, y) for x, n, y in zip(wd, ns, yf_fused)], k, producer, a, b, w, eps)
    q8.q8_check()
    y_two = [nan_f32(n) for n in ns]
    row = _two_launch(q8, producer, k, a, b, w, eps, [(x, n, y) for x, n, y in zip(wd, ns, y_two)])
    qs_r, ds_r = oracle.quantize(host(row).reshape(1, k), 1)
    for blob, n, yf, yt in zip(blobs, ns, yf_fused, y_two):
        assert torch.equal(yf, yt), f"producer {producer} {n}x{k}: fused != two launches"
        yr, ar = oracle.gemv(blob, n, k, qs_r, ds_r)
        assert_gemm_close(host(yf), yr, ar, f"fused producer {producer} {n}x{k}")


@pytest.mark.parametrize("producer", [1, 2])
def test_fused_subnormal_scales_equal_two_launches(q8, producer):
    """Activations whose blocks have subnormal d (the clamp decides codes):
    the fused prologue's plane equals the standalone producer's."""
    import torch

    from .test_parity_quantize_gpu import _tiny_rows

    k, ns = 3584, [300, 64]
    if producer == 1:  # the activation itself has subnormal block scales
        a_h, w_h = _tiny_rows(1, k, 7)[0], None
    else:              # a norm weight that makes every normalized value subnormal
        a_h = syn.activations(syn.rng(72, k), 1, k)[0]
        w_h = np.full(k, 1e-38, np.float32)
    a = dev(a_h)
    w = dev(w_h) if w_h is not None else None
    blobs = [_weights(20 + i, n, k) for i, n in enumerate(ns)]
    wd = [dev(bl) for bl in blobs]
    yf = [nan_f32(n) for n in ns]
    q8.q8_0_gemv_fused([(x, n, y) for x, n, y in zip(wd, ns, yf)], k, producer, a, None, w, 1e-6)
    q8.q8_check()
    yt = [nan_f32(n) for n in ns]
    _two_launch(q8, producer, k, a, None, w, 1e-6, [(x, n, y) for x, n, y in zip(wd, ns, yt)])
    for n, f, t in zip(ns, yf, yt):
        assert torch.equal(f, t), f"producer {producer} {n}x{k}: fused != two launches"


def test_fused_rmsnorm_zero_row(q8):
    """An all-zero row: the scale is rsqrt(eps), every code and d is 0, every output exactly 0."""
    k, n = 3584, 300
    blob = _weights(5, n, k)
    y = nan_f32(n)
    import torch

    x = torch.zeros(k, dtype=torch.float32, device="cuda")
    w = torch.ones(k, dtype=torch.float32, device="cuda")
    q8.q8_0_gemv_fused([(dev(blob), n, y)], k, q8.PRODUCER_RMSNORM, x, None, w, 1e-6)
    q8.q8_check()
    assert (host(y) == 0).all()


def test_fused_rejects_unsupported(q8):
    import torch

    k = 2080  # 65 blocks: not a multiple of 8 blocks (the staged path only)
    w = torch.zeros(34 * (k // 32), dtype=torch.uint8, device="cuda")
    y = torch.zeros(1, dtype=torch.float32, device="cuda")
    x = torch.zeros(k, dtype=torch.float32, device="cuda")
    with pytest.raises(q8.Q8Error):
        q8.q8_0_gemv_fused([(w, 1, y)], k, q8.PRODUCER_QUANT, x)
    k = 256
    w = torch.zeros(34 * (k // 32), dtype=torch.uint8, device="cuda")
    x = torch.zeros(k, dtype=torch.float32, device="cuda")
    with pytest.raises(q8.Q8Error):
        q8.q8_0_gemv_fused([(w, 1, y)], k, 4, x)          # no such producer
    with pytest.raises(q8.Q8Error):
        q8.q8_0_gemv_fused([(w, 1, y)], k, q8.PRODUCER_SWIGLU, x)   # up missing
    with pytest.raises(q8.Q8Error):
        q8.q8_0_gemv_fused([(w, 1, y)], k, q8.PRODUCER_RMSNORM, x)  # weight missing


GATE_UP = [
    # (nf, k): the model's shape, a ragged number of 64-row units per CTA, long rows (several pieces), the k limits
    (18944, 3584),
    (96, 2304),
    (4096, 18944),
    (1024, 65536),
    (32, 4096),
]


@pytest.mark.parametrize("producer", [0, 1, 2])
@pytest.mark.parametrize("nf,k", GATE_UP)
def test_gate_up_equals_grouped_then_swiglu_quant(q8, producer, nf, k):
    """q8_0_gemv_gate_up: its gate/up outputs bit for bit those of the grouped GEMV (or the fused one) on the same
    activation, its plane bit for bit swiglu_quant's encoding of those outputs, and that plane within the oracle's
    pinned arithmetic (oracle.quantize of the f32 SwiGLU row the standalone kernel writes)."""
    import torch

    if producer == 2 and k > 32768:
        pytest.skip("RMSNorm rows are limited to 32768")
    wg_h, wu_h = _weights(20, nf, k), _weights(21, nf, k)
    wg, wu = dev(wg_h), dev(wu_h)
    a_h, _, w_h = _inputs(producer or 1, k, 7)
    a, nw = dev(a_h), (dev(w_h) if w_h is not None else None)
    eps = 1e-6
    qs, ds = q8.empty_plane(1, k)
    q8.quantize_q8_0(a.view(1, k), qs, ds)
    q_out, d_out = q8.empty_plane(1, nf)
    q_out.fill_(-91), d_out.fill_(0x5A5A5A5A)
    yg, yu = nan_f32(nf), nan_f32(nf)
    if producer == 0:
        q8.q8_0_gemv_gate_up(wg, wu, nf, k, q_out, d_out, qs=qs, ds=ds, y_gate=yg, y_up=yu)
    else:
        q8.q8_0_gemv_gate_up(wg, wu, nf, k, q_out, d_out, producer=producer, a=a, norm_w=nw, eps=eps,
                             y_gate=yg, y_up=yu)
    q8.q8_check()
    # the same projections the plain way
    rg, ru = nan_f32(nf), nan_f32(nf)
    if producer == 0:
        q8.q8_0_gemv_grouped([(wg, nf, rg), (wu, nf, ru)], k, qs, ds)
    else:
        q8.q8_0_gemv_fused([(wg, nf, rg), (wu, nf, ru)], k, producer, a, None, nw, eps)
    q8.q8_check()
    assert torch.equal(yg, rg) and torch.equal(yu, ru), "gate/up outputs differ from the grouped GEMV"
    ys = nan_f32(1, nf)
    q_ref, d_ref = q8.empty_plane(1, nf)
    q8.swiglu_quant(rg.view(1, nf), ru.view(1, nf), ys, q_ref, d_ref)
    q8.q8_check()
    assert torch.equal(q_out, q_ref) and torch.equal(d_out, d_ref), "plane differs from swiglu_quant's"
    qo, do = oracle.quantize(host(ys), 1)
    assert np.array_equal(host(q_out), qo) and np.array_equal(host(d_out).view(np.uint32), do)


def test_gate_up_without_f32_outputs(q8):
    """y_gate / y_up may be NULL: the plane is the same bytes."""
    import torch

    nf, k = 18944, 3584
    wg, wu = dev(_weights(22, nf, k)), dev(_weights(23, nf, k))
    a = dev(_inputs(1, k, 8)[0])
    q1, d1 = q8.empty_plane(1, nf)
    q2, d2 = q8.empty_plane(1, nf)
    yg, yu = nan_f32(nf), nan_f32(nf)
    q8.q8_0_gemv_gate_up(wg, wu, nf, k, q1, d1, producer=1, a=a, y_gate=yg, y_up=yu)
    q8.q8_0_gemv_gate_up(wg, wu, nf, k, q2, d2, producer=1, a=a)
    q8.q8_check()
    assert torch.equal(q1, q2) and torch.equal(d1, d2)


def test_fused_decode_pair_full_size(q8):
    """The decode step's launch at full size: quantize inside the grouped 12288 x 7168 + 96 x 7168 GEMV, on an
    activation with the decode recipe (N(0, 1.5), 1 % outliers x20); every output against the two-launch path
    (bit for bit) and the oracle."""
    import torch

    k, ns = 7168, (12288, 96)
    g = syn.rng(72, k)
    x_h = syn.activations(g, 1, k, sigma=1.5, outlier_frac=0.01, outlier_mult=20.0)[0]
    x = dev(x_h)
    blobs = [_weights(30 + i, n, k) for i, n in enumerate(ns)]
    wd = [dev(b) for b in blobs]
    yf = [nan_f32(n) for n in ns]
    q8.q8_0_gemv_fused([(w, n, y) for w, n, y in zip(wd, ns, yf)], k, q8.PRODUCER_QUANT, x)
    q8.q8_check()
    yt = [nan_f32(n) for n in ns]
    qs, ds = q8.empty_plane(q8.q8_plane_rows(1), k)
    q8.quantize_q8_0(x.view(1, k), qs, ds)
    q8.q8_0_gemv_grouped([(w, n, y) for w, n, y in zip(wd, ns, yt)], k, qs, ds)
    q8.q8_check()
    qr, dr = oracle.quantize(x_h.reshape(1, k), 1)
    for blob, n, a, b in zip(blobs, ns, yf, yt):
        assert torch.equal(a, b), f"{n}x{k}: fused != two launches"
        yr, ar = oracle.gemv(blob, n, k, qr, dr)
        assert_gemm_close(host(a), yr, ar, f"fused decode {n}x{k}")
