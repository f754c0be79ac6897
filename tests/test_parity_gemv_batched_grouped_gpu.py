"""GPU parity of the grouped small-batch projection (q8_0_gemv_batched_grouped)
against the oracle and against the single-projection call.

Several projections of the same plane rows (a layer's Q, K and V, or its gate
and up) form one launch: each projection's outputs are the GEMM formula
Y[t][i] = sum_b d_w * d_a * isum ("12 - r5-r6 re-ranking + structural rewrite
spec", sec. 2) over its own rows, and "Part 4 - Lecture 05", sec. 2.5 is the
one-launch-per-activation rule this applies.  Outputs are NaN-poisoned and
compared with the oracle's fp64 values within the GEMM tolerance; the
exact-epilogue configuration (every f32 operation exact) is compared bit for
bit, whatever split of k the launch picks.  A group of one projection is the
single call (the same grid and split): bit for bit.  Shapes cover ragged
row counts (a projection whose last 128-row tile is partly empty, one
smaller than a tile), both token tiles (t <= 8 and 9..16), the largest group,
and k/32 not a multiple of 8 (the generic kernel, one projection at a time).
"""
import numpy as np
import pytest

import oracle

from ._parity import assert_gemm_close, dev, host, nan_f32
from .test_parity_gemv_gemm_gpu import _plane, _weights

pytestmark = pytest.mark.gpu

GROUPS = [
    (3584, (3584, 512, 512), 16),              # a 7B layer's Q, K, V at the decode batch
    (3584, (18944, 18944), 9),                 # its gate and up
    (1024, (37, 1000, 4099), 5),               # ragged tiles; one projection smaller than a tile
    (2048, (300,), 12),                        # a group of one
    (512, (129, 64, 200, 32, 777, 1, 300, 96), 16),  # the largest group
    (96, (513, 40), 7),                        # k/32 = 3: generic kernel per projection
]


def _run(q8, k, blobs, ns, qs, ds, t):
    ys = [nan_f32(t, n) for n in ns]
    q8.q8_0_gemv_batched_grouped([(dev(b), n, y) for b, n, y in zip(blobs, ns, ys)], k, dev(qs),
                                 dev(ds.view(np.int32)), t)
    q8.q8_check()
    return ys


@pytest.mark.parametrize("k,ns,t", GROUPS)
def test_gemv_batched_grouped_matches_oracle(q8, k, ns, t):
    import torch

    blobs = [_weights(70 + i, n, k) for i, n in enumerate(ns)]
    qs, ds = _plane(70, t, k, rows_pad=128)
    ys = _run(q8, k, blobs, ns, qs, ds, t)
    for i, (blob, n, y) in enumerate(zip(blobs, ns, ys)):
        assert not torch.isnan(y).any().item(), f"projection {i}: unwritten outputs"
        if n * k > 4096 * 4096:  # the oracle on sampled rows for the wide projections
            ni = np.unique(np.concatenate([[0, n - 1], np.random.default_rng(n).integers(0, n, 96)]))
        else:
            ni = np.arange(n)
        yr, ar = oracle.gemm(blob, n, k, qs, ds, t_idx=np.arange(t), n_idx=ni)
        assert_gemm_close(host(y)[:, ni], yr, ar, f"grouped batched {i}: {n}x{k} t={t}")


@pytest.mark.parametrize("k,ns,t", [(2048, (300, 64, 1000), 16), (1024, (129, 7), 3), (18944, (64, 512), 9)])
def test_gemv_batched_grouped_exact_epilogue_bit_equal(q8, k, ns, t):
    blobs = [_weights(80 + i, n, k, exact=True) for i, n in enumerate(ns)]
    qs, ds = _plane(80, t, k, exact=True)
    ys = _run(q8, k, blobs, ns, qs, ds, t)
    for blob, n, y in zip(blobs, ns, ys):
        yr, _ = oracle.gemm(blob, n, k, qs, ds, t_idx=np.arange(t))
        assert np.array_equal(host(y).astype(np.float64), yr), f"{n}x{k} t={t}"


@pytest.mark.parametrize("n,k,t", [(3584, 3584, 16), (1000, 2048, 5), (37, 512, 1)])
def test_group_of_one_is_the_single_call(q8, n, k, t):
    import torch

    blob = _weights(90, n, k)
    qs, ds = _plane(90, t, k, rows_pad=128)
    (y_grp,) = _run(q8, k, [blob], [n], qs, ds, t)
    y_one = nan_f32(t, n)
    q8.q8_0_gemv_batched(dev(blob), n, k, dev(qs), dev(ds.view(np.int32)), t, y_one)
    q8.q8_check()
    assert torch.equal(y_grp, y_one)


def test_gemv_batched_grouped_deterministic(q8):
    import torch

    k, ns, t = 3584, (3584, 512, 512), 16
    blobs = [_weights(91 + i, n, k) for i, n in enumerate(ns)]
    qs, ds = _plane(91, t, k, rows_pad=128)
    first = _run(q8, k, blobs, ns, qs, ds, t)
    for _ in range(2):
        again = _run(q8, k, blobs, ns, qs, ds, t)
        assert all(torch.equal(a, b) for a, b in zip(first, again))


def test_gemv_batched_grouped_rejects_bad_arguments(q8):
    import torch

    k = 256
    w = torch.zeros(8 * (k // 32) * 34, dtype=torch.uint8, device="cuda")
    qs = torch.zeros(128, k, dtype=torch.int8, device="cuda")
    ds = torch.zeros(128, k // 32, dtype=torch.int32, device="cuda")
    y = torch.zeros(17 * 8, dtype=torch.float32, device="cuda")
    for t in (0, 17):
        with pytest.raises(q8.Q8Error):
            q8.q8_0_gemv_batched_grouped([(w, 8, y)], k, qs, ds, t)
    with pytest.raises(ValueError):
        q8.q8_0_gemv_batched_grouped([(w, 8, y)] * 9, k, qs, ds, 4)


@pytest.mark.parametrize("case", range(6))
def test_gemv_batched_grouped_random_groups(q8, case):
    """Seeded random groups: 1..8 projections of 1..5000 rows, k a multiple of
    256 up to 4096 (or 96 for the generic kernel), 1..16 tokens."""
    import torch

    g = np.random.default_rng(1000 + case)
    count = int(g.integers(1, 9))
    k = 96 if case == 5 else 256 * int(g.integers(1, 17))
    t = int(g.integers(1, 17))
    ns = [int(g.integers(1, 5001)) for _ in range(count)]
    blobs = [_weights(200 + 10 * case + i, n, k) for i, n in enumerate(ns)]
    qs, ds = _plane(200 + case, t, k, rows_pad=128)
    ys = _run(q8, k, blobs, ns, qs, ds, t)
    for i, (blob, n, y) in enumerate(zip(blobs, ns, ys)):
        assert not torch.isnan(y).any().item(), f"projection {i}: unwritten outputs"
        yr, ar = oracle.gemm(blob, n, k, qs, ds, t_idx=np.arange(t))
        assert_gemm_close(host(y), yr, ar, f"random group {case}, projection {i}: {n}x{k} t={t}")
