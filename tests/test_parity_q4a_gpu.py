"""GPU parity of q4a_gemv (asymmetric 4-bit weight blocks, value d*nib - m)
against the oracle.

Per block the kernel adds d*d_a*isum and -m*d_a*ssum, the min term taken from
the plane's int16 block sum ("54 - r51 - producer-fused A-quantize mode 1",
sec. 2.1).  Outputs are NaN-poisoned first and compared with the oracle's
fp64 value within 1e-5 * sum_b (|d*d_a*isum| + |m*d_a*ssum|); the
exact-epilogue configuration (power-of-two scales and mins, small codes:
every f32 operation exact in any order) requires bit equality, which checks
the nibble unpacking, the dp4a pairing of nibble halves with activation words
and the sign and source of the min term.  Shapes cover one chunk per row
(k = 128, 32 rows per warp), ragged row counts, rows spanning several lanes'
chunk pairs and an odd trailing chunk, and the full-size decode projection.
Rows of at most 512 chunks (k <= 65536) run on the staged kernel (per-warp
rings of bulk-copied pieces); longer rows on the wide kernel (weights loaded
straight into registers): both sides of that boundary are covered.
"""
import numpy as np
import pytest

import oracle
from int8_quantized_projection_gb300 import synthetic as syn

from ._parity import assert_gemm_close, dev, host, nan_f32

pytestmark = pytest.mark.gpu


def _weights(seed, n, k, exact=False):
    g = syn.rng(80, seed, n, k)
    blob, d16, m16, nib = syn.q4a_weights(g, n, k)
    if exact:
        e = g.integers(-4, -1, size=d16.shape)
        d16 = (2.0 ** e).astype(np.float16).view(np.uint16)
        em = g.integers(-3, 0, size=m16.shape)
        m16 = (2.0 ** em).astype(np.float16).view(np.uint16)
        blob = syn.pack_q4a(d16, m16, nib)
    return blob


def _plane(seed, k, exact=False):
    g = syn.rng(81, seed, k)
    if exact:
        qa = g.integers(-3, 4, size=(1, k)).astype(np.int8)
        e = g.integers(-4, -1, size=(1, k // 32))
        d16 = (2.0 ** e).astype(np.float16).view(np.uint16)
        ssum = qa.reshape(1, k // 32, 32).astype(np.int64).sum(-1)
        ds = d16.astype(np.uint32) | (ssum.astype(np.int16).view(np.uint16).astype(np.uint32) << 16)
        return qa, ds
    return oracle.quantize(syn.activations(g, 1, k, sigma=1.5, outlier_frac=0.01))


def _run(q8, blob, n, k, qs, ds):
    y = nan_f32(n)
    q8.q4a_gemv(dev(blob), n, k, dev(qs), dev(ds.view(np.int32)), y)
    q8.q8_check()
    return y


SHAPES = [
    (256, 128),      # one chunk per row: 32 rows per warp
    (1000, 512),     # 4 chunks per row
    (333, 1152),     # 9 chunks: lane pairs plus an odd trailing chunk
    (1001, 2048),    # 16 chunks, ragged n
    (77, 18944),     # 148 chunks: rows spanning many chunk pairs
    (3, 256), (1, 128),
    (4099, 7168),    # ragged n, 56 chunks
    (12288, 7168),   # full-size decode projection
    (40, 65536),     # 512 chunks: the longest row of the staged kernel
    (50, 65664),     # 513 chunks: the wide kernel
    (9, 131072),     # 1024 chunks, wide kernel
]


@pytest.mark.parametrize("n,k", SHAPES)
def test_q4a_gemv_matches_oracle(q8, n, k):
    blob = _weights(1, n, k)
    qs, ds = _plane(1, k)
    y = _run(q8, blob, n, k, qs, ds)
    yr, ar = oracle.q4a_gemv(blob, n, k, qs, ds)
    assert_gemm_close(host(y), yr, ar, f"q4a_gemv {n}x{k}")


@pytest.mark.parametrize("n,k", [(300, 2048), (77, 18944), (512, 128), (129, 7168), (33, 65536), (21, 65664)])
def test_q4a_gemv_exact_epilogue_bit_equal(q8, n, k):
    blob = _weights(2, n, k, exact=True)
    qs, ds = _plane(2, k, exact=True)
    y = _run(q8, blob, n, k, qs, ds)
    yr, _ = oracle.q4a_gemv(blob, n, k, qs, ds)
    assert np.array_equal(host(y).astype(np.float64), yr)


def test_q4a_gemv_deterministic(q8):
    import torch

    n, k = 12288, 7168
    blob = dev(_weights(3, n, k))
    qs, ds = _plane(3, k)
    qs, ds = dev(qs), dev(ds.view(np.int32))
    outs = []
    for _ in range(3):
        y = nan_f32(n)
        q8.q4a_gemv(blob, n, k, qs, ds, y)
        q8.q8_check()
        outs.append(y.clone())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


def test_q4a_decode_chain_from_the_gpu_plane(q8):
    """quantize_q8_0 on the GPU, then q4a_gemv on that plane: the oracle applied to the
    GPU's own plane (itself checked bit-exact elsewhere) agrees."""
    n, k = 3584, 18944
    g = syn.rng(82, 0)
    x = syn.activations(g, 1, k)
    qs, ds = q8.empty_plane(1, k)
    q8.quantize_q8_0(dev(x), qs, ds)
    blob = _weights(4, n, k)
    y = nan_f32(n)
    q8.q4a_gemv(dev(blob), n, k, qs, ds, y)
    q8.q8_check()
    yr, ar = oracle.q4a_gemv(blob, n, k, host(qs), host(ds).view(np.uint32))
    assert_gemm_close(host(y), yr, ar, "q4a decode chain")


# ---------------------------------------------------------------------------
# q4a_gemv_batched: t = 2..16 tokens, the weights read once for all of them
# (t <= 8: one token tile on the int8 MMA; t > 8: two tiles on the f16 MMA).
# ---------------------------------------------------------------------------
def _plane_t(seed, t, k, exact=False):
    """Plane rows [0, t) of t tokens, padded to 128 rows (rows >= t zero)."""
    g = syn.rng(83, seed, t, k)
    if exact:
        qa = np.zeros((128, k), np.int8)
        qa[:t] = g.integers(-3, 4, size=(t, k)).astype(np.int8)
        e = g.integers(-4, -1, size=(128, k // 32))
        d16 = (2.0 ** e).astype(np.float16).view(np.uint16)
        ssum = qa.reshape(128, k // 32, 32).astype(np.int64).sum(-1)
        ds = d16.astype(np.uint32) | (ssum.astype(np.int16).view(np.uint16).astype(np.uint32) << 16)
        ds[t:] = 0
        return qa, ds
    return oracle.quantize(syn.activations(g, t, k, sigma=1.5, outlier_frac=0.01), 128)


def _run_batched(q8, blob, n, k, qs, ds, t):
    y = nan_f32(t, n)
    q8.q4a_gemv_batched(dev(blob), n, k, dev(qs), dev(ds.view(np.int32)), t, y)
    q8.q8_check()
    return y


BATCHED = [
    (256, 256, 2),     # one 8-block piece per row
    (1000, 512, 5),    # ragged row tile, one token tile
    (333, 2048, 8),
    (77, 18944, 9),    # two token tiles (f16 MMA), long rows split over a cluster
    (4099, 7168, 16),  # ragged n, full tile pair
    (3, 256, 3),
    (12288, 7168, 16), # full-size decode projection
]


@pytest.mark.parametrize("n,k,t", BATCHED)
def test_q4a_gemv_batched_matches_oracle(q8, n, k, t):
    blob = _weights(5, n, k)
    qs, ds = _plane_t(5, t, k)
    y = _run_batched(q8, blob, n, k, qs, ds, t)
    yr, ar = oracle.q4a_gemm(blob, n, k, qs, ds, t_idx=np.arange(t))
    assert_gemm_close(host(y), yr, ar, f"q4a_gemv_batched {n}x{k} t={t}")


@pytest.mark.parametrize("n,k,t", [(300, 2048, 7), (129, 7168, 16), (77, 18944, 4)])
def test_q4a_gemv_batched_exact_epilogue_bit_equal(q8, n, k, t):
    blob = _weights(6, n, k, exact=True)
    qs, ds = _plane_t(6, t, k, exact=True)
    y = _run_batched(q8, blob, n, k, qs, ds, t)
    yr, _ = oracle.q4a_gemm(blob, n, k, qs, ds, t_idx=np.arange(t))
    assert np.array_equal(host(y).astype(np.float64), yr)


def test_q4a_gemv_batched_one_token_is_q4a_gemv(q8):
    n, k = 1001, 2048
    blob = _weights(7, n, k)
    qs, ds = _plane(7, k)
    y1 = _run_batched(q8, blob, n, k, qs, ds, 1)
    y = _run(q8, blob, n, k, qs, ds)
    assert np.array_equal(host(y1).reshape(-1), host(y))


def test_q4a_gemv_batched_ignores_plane_rows_past_t(q8):
    """Rows at and past t hold garbage: the result is unchanged (they arrive
    as zeros only through the tensor map's bounds, never from the plane)."""
    n, k, t = 500, 2048, 6
    blob = _weights(8, n, k)
    qs, ds = _plane_t(8, t, k)
    y = _run_batched(q8, blob, n, k, qs, ds, t)
    g = syn.rng(84, 0)
    qs2, ds2 = qs.copy(), ds.copy()
    qs2[t:] = g.integers(-127, 128, size=qs2[t:].shape).astype(np.int8)
    ds2[t:] = g.integers(0, 2**31, size=ds2[t:].shape).astype(np.uint32)
    y2 = _run_batched(q8, blob, n, k, qs2, ds2, t)
    assert np.array_equal(host(y), host(y2))


def test_q4a_gemv_batched_deterministic(q8):
    import torch

    n, k, t = 12288, 7168, 12
    blob = dev(_weights(9, n, k))
    qs, ds = _plane_t(9, t, k)
    qs, ds = dev(qs), dev(ds.view(np.int32))
    outs = []
    for _ in range(3):
        y = nan_f32(t, n)
        q8.q4a_gemv_batched(blob, n, k, qs, ds, t, y)
        q8.q8_check()
        outs.append(y.clone())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


# ---------------------------------------------------------------------------
# q4a_gemv_batched_grouped: several projections of the same plane rows in one
# launch (the small-batch kernel over their joined row tiles; one token: the
# batch-1 kernel projection by projection)
# ---------------------------------------------------------------------------
def _run_grouped(q8, k, blobs, ns, qs, ds, t):
    ys = [nan_f32(t, n) for n in ns]
    q8.q4a_gemv_batched_grouped([(dev(b), n, y) for b, n, y in zip(blobs, ns, ys)], k, dev(qs),
                                dev(ds.view(np.int32)), t)
    q8.q8_check()
    return ys


@pytest.mark.parametrize("k,ns,t", [(3584, (3584, 512, 512), 16), (1024, (37, 1000, 300), 5),
                                    (2048, (129, 64, 700, 1, 256, 96, 33, 512), 12), (512, (300, 77), 1)])
def test_q4a_gemv_batched_grouped_matches_oracle(q8, k, ns, t):
    import torch

    blobs = [_weights(50 + i, n, k) for i, n in enumerate(ns)]
    qs, ds = _plane_t(50, t, k)
    ys = _run_grouped(q8, k, blobs, ns, qs, ds, t)
    for i, (blob, n, y) in enumerate(zip(blobs, ns, ys)):
        assert not torch.isnan(y).any().item(), f"projection {i}: unwritten outputs"
        yr, ar = oracle.q4a_gemm(blob, n, k, qs, ds, t_idx=np.arange(t))
        assert_gemm_close(host(y), yr, ar, f"q4a grouped {i}: {n}x{k} t={t}")


def test_q4a_gemv_batched_grouped_exact_epilogue_bit_equal(q8):
    k, ns, t = 2048, (300, 64, 129), 9
    blobs = [_weights(60 + i, n, k, exact=True) for i, n in enumerate(ns)]
    qs, ds = _plane_t(60, t, k, exact=True)
    ys = _run_grouped(q8, k, blobs, ns, qs, ds, t)
    for blob, n, y in zip(blobs, ns, ys):
        yr, _ = oracle.q4a_gemm(blob, n, k, qs, ds, t_idx=np.arange(t))
        assert np.array_equal(host(y).astype(np.float64), yr)


@pytest.mark.parametrize("t", [1, 6, 16])
def test_q4a_group_of_one_is_the_single_call(q8, t):
    import torch

    n, k = 1000, 2048
    blob = _weights(70, n, k)
    qs, ds = _plane_t(70, t, k)
    (y_grp,) = _run_grouped(q8, k, [blob], [n], qs, ds, t)
    y_one = _run_batched(q8, blob, n, k, qs, ds, t)
    assert torch.equal(y_grp, y_one)
