"""GPU parity of the small-batch projection (q8_0_gemv_batched, and q8_0_gemm
for t <= 16, which hands those calls to it) against the oracle.

The contraction is the GEMM's, Y[t][i] = sum_b d_w * d_a * isum ("12 - r5-r6
re-ranking + structural rewrite spec", sec. 2), for 1..16 tokens.  Outputs
are NaN-poisoned before the call, compared with the oracle's fp64 value
within 1e-5 * sum_b |term_b|, and the exact-epilogue configuration (every f32
operation exact) requires bit equality, which checks the tensor-core integer
block dot products, the k permutation inside a block and the fragment
layouts.  Shapes cover: token counts on both sides of the 8-token tile (1, 2,
7, 8, 9, 15, 16), row counts that leave a ragged last 32-row CTA, k with 1..4
groups of 8 blocks per warp (and warps with none), k/32 not a multiple of 8
(generic kernel), and the decode-batch shapes of the 28-layer stack at t = 16
(full size, sampled rows).
"""
import numpy as np
import pytest

import oracle
from int8_quantized_projection_gb300 import synthetic as syn

from ._parity import assert_gemm_close, dev, host, nan_f32
from .test_parity_gemv_gemm_gpu import _plane, _weights

pytestmark = pytest.mark.gpu


def _run(q8, entry, blob, n, k, qs, ds, t):
    y = nan_f32(t, n)
    getattr(q8, entry)(dev(blob), n, k, dev(qs), dev(ds.view(np.int32)), t, y)
    q8.q8_check()
    return y


SHAPES = [
    (32, 256, 2),      # one CTA, one 8-block group: warps 1..3 have no k range
    (37, 512, 7),      # ragged last CTA (5 rows), two groups
    (100, 1024, 8),    # 4 groups: one per warp
    (1000, 2048, 9),   # second token tile, 8 groups
    (257, 3584, 15),   # 14 groups (uneven split over 4 warps)
    (4099, 7168, 16),  # 28 groups, ragged n
    (64, 18944, 16),   # 74 groups per row
    (513, 96, 5),      # k/32 = 3: generic kernel
    (300, 2048, 1),    # a single token
]


@pytest.mark.parametrize("n,k,t", SHAPES)
def test_gemv_batched_matches_oracle(q8, n, k, t):
    blob = _weights(20, n, k)
    qs, ds = _plane(20, t, k, rows_pad=((t + 127) // 128) * 128)
    y = host(_run(q8, "q8_0_gemv_batched", blob, n, k, qs, ds, t))
    yr, ar = oracle.gemm(blob, n, k, qs, ds, t_idx=np.arange(t))
    assert_gemm_close(y, yr, ar, f"gemv_batched {n}x{k} t={t}")


@pytest.mark.parametrize("n,k,t", [(300, 2048, 16), (77, 18944, 9), (129, 7168, 3), (64, 256, 8)])
def test_gemv_batched_exact_epilogue_bit_equal(q8, n, k, t):
    blob = _weights(21, n, k, exact=True)
    qs, ds = _plane(21, t, k, exact=True)
    y = host(_run(q8, "q8_0_gemv_batched", blob, n, k, qs, ds, t))
    yr, _ = oracle.gemm(blob, n, k, qs, ds)
    assert np.array_equal(y.astype(np.float64), yr)


def test_gemv_batched_ignores_plane_rows_past_t(q8):
    """Rows t..rows_pad-1 of the plane hold garbage; the result must not depend on them."""
    import torch

    n, k, t = 200, 2048, 5
    blob = _weights(22, n, k)
    qs, ds = _plane(22, t, k, rows_pad=128)
    y0 = _run(q8, "q8_0_gemv_batched", blob, n, k, qs, ds, t)
    g = syn.rng(22, 1)
    qs2, ds2 = qs.copy(), ds.copy()
    qs2[t:] = g.integers(-127, 128, size=qs2[t:].shape).astype(np.int8)
    ds2[t:] = g.integers(0, 2**32, size=ds2[t:].shape, dtype=np.uint64).astype(np.uint32)
    y1 = _run(q8, "q8_0_gemv_batched", blob, n, k, qs2, ds2, t)
    assert torch.equal(y0, y1)


@pytest.mark.parametrize("n,k,t", [(1000, 3584, 12), (4099, 7168, 16), (513, 96, 5), (300, 2048, 1)])
def test_gemm_small_t_is_the_batched_path(q8, n, k, t):
    """q8_0_gemm with t <= 16 gives bit-identical results to q8_0_gemv_batched (t == 1: q8_0_gemv)."""
    import torch

    blob = _weights(23, n, k)
    qs, ds = _plane(23, t, k, rows_pad=128)
    y_gemm = _run(q8, "q8_0_gemm", blob, n, k, qs, ds, t)
    if t == 1:
        y_ref = nan_f32(n)
        q8.q8_0_gemv(dev(blob), n, k, dev(qs), dev(ds.view(np.int32)), y_ref)
        q8.q8_check()
        y_ref = y_ref.view(1, n)
    else:
        y_ref = _run(q8, "q8_0_gemv_batched", blob, n, k, qs, ds, t)
    assert torch.equal(y_gemm, y_ref)


def test_gemv_batched_deterministic(q8):
    import torch

    n, k, t = 12288, 7168, 16
    blob = dev(_weights(24, n, k))
    qs, ds = _plane(24, t, k, rows_pad=128)
    qs, ds = dev(qs), dev(ds.view(np.int32))
    outs = []
    for _ in range(3):
        y = nan_f32(t, n)
        q8.q8_0_gemv_batched(blob, n, k, qs, ds, t, y)
        q8.q8_check()
        outs.append(y.clone())
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])


# the projections of the 28-layer stack (q/o 3584x3584, k/v 512x3584, gate/up
# 18944x3584, down 3584x18944) and the 152064-row lm_head, at t = 16
@pytest.mark.parametrize("n,k", [(3584, 3584), (512, 3584), (18944, 3584), (3584, 18944), (152064, 3584)])
def test_gemv_batched_full_size_sampled(q8, n, k):
    import torch

    t = 16
    blob = _weights(25, n, k)
    qs, ds = _plane(25, t, k, rows_pad=128)
    y = _run(q8, "q8_0_gemv_batched", blob, n, k, qs, ds, t)
    assert not torch.isnan(y).any().item(), "unwritten outputs"
    g = syn.rng(63, n, k, t)
    ni = np.unique(np.concatenate([[0, n - 1, (n // 32) * 32 - 1], g.integers(0, n, 128)]))
    yr, ar = oracle.gemm(blob, n, k, qs, ds, t_idx=np.arange(t), n_idx=ni)
    assert_gemm_close(host(y)[:, ni], yr, ar, f"gemv_batched {n}x{k} t={t} (sampled)")


def test_gemv_batched_rejects_bad_token_counts(q8):
    import torch

    blob = torch.zeros(8 * 8 * 34, dtype=torch.uint8, device="cuda")
    qs = torch.zeros(128, 256, dtype=torch.int8, device="cuda")
    ds = torch.zeros(128, 8, dtype=torch.int32, device="cuda")
    y = torch.zeros(17 * 8, dtype=torch.float32, device="cuda")
    for t in (0, 17):
        with pytest.raises(q8.Q8Error):
            q8.q8_0_gemv_batched(blob, 8, 256, qs, ds, t, y)
