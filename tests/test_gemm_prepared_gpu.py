"""The prefill GEMM on prepared weights (q8_0_gemm_prepare_weights once per
matrix, then q8_0_gemm_prepared per call) against q8_0_gemm and the oracle.

The prepared form is the output of the weight pre-pass that q8_0_gemm runs
on every call (the codes widened to f16, exactly; each block's d_w as f32).
The GEMM on it runs the same kernels on the same operands, so its output
must equal q8_0_gemm's bit for bit, on every tcgen05 shape (unsplit, split
over k, short k); at unit scales with full-range codes it must also equal
the oracle's integer sums exactly, and on realistic data stay within the
GEMM tolerance of the oracle.  Calls that take the other paths (t <= 64,
(k/32) % 8 != 0) read the Q8_0 weights and behave as q8_0_gemm does.

Sources: the per-block scale correction ("12 - r5-r6 re-ranking +
structural rewrite spec", sec. 2 and 3.1) and the q8_0 plane ("54 - r51 -
producer-fused A-quantize mode 1", sec. 2.1).
"""
import numpy as np
import pytest

import oracle
from int8_quantized_projection_gb300 import synthetic as syn

from ._parity import assert_gemm_close, dev, host, nan_f32
from .test_parity_exact_full_range_gpu import _assert_exact, _unit_plane, _unit_weights

pytestmark = pytest.mark.gpu

TC_CASES = [
    (512, 1024, 65),     # split over k (few tiles)
    (256, 1024, 300),    # split over k
    (2048, 1024, 1536),  # unsplit (16 x 8 tiles)
    (1000, 256, 400),    # short k
    (300, 2048, 777),    # ragged rows and tokens
]


def _plane(seed, t, k):
    g = syn.rng(95, seed, t, k)
    x = syn.activations(g, t, k, sigma=1.5, outlier_frac=0.01)
    rows_pad = ((t + 127) // 128) * 128
    qs, ds = oracle.quantize(x, rows_pad)
    return qs, ds


@pytest.mark.parametrize("n,k,t", TC_CASES)
def test_prepared_equals_plain_and_oracle(q8, n, k, t):
    import torch

    blob = syn.q8_0_weights(syn.rng(96, n, k), n, k)[0]
    qs, ds = _plane(1, t, k)
    w, qd, dd = dev(blob), dev(qs), dev(ds.view(np.int32))
    wprep = q8.q8_0_gemm_prepare_weights(w, n, k)
    assert wprep.numel() == q8.q8_0_gemm_prepared_weights_bytes(n, k)
    y_plain, y_prep = nan_f32(t, n), nan_f32(t, n)
    q8.q8_0_gemm(w, n, k, qd, dd, t, y_plain)
    q8.q8_0_gemm_prepared(None, wprep, n, k, qd, dd, t, y_prep)
    q8.q8_check()
    assert torch.equal(y_plain, y_prep), f"{n}x{k} t={t}: prepared differs from the per-call pre-pass"
    yr, ar = oracle.gemm(blob, n, k, qs, ds, t_idx=np.arange(t))
    assert_gemm_close(host(y_prep), yr, ar, f"prepared {n}x{k} t={t}")


@pytest.mark.parametrize("n,k,t", [(512, 1024, 65), (256, 1024, 300), (2048, 1024, 1536), (1000, 256, 400)])
def test_prepared_full_range_bit_exact(q8, n, k, t):
    blob = _unit_weights(41, n, k)
    qs, ds = _unit_plane(41, t, k, rows_pad=((t + 127) // 128) * 128)
    wprep = q8.q8_0_gemm_prepare_weights(dev(blob), n, k)
    y = nan_f32(t, n)
    q8.q8_0_gemm_prepared(None, wprep, n, k, dev(qs), dev(ds.view(np.int32)), t, y)
    q8.q8_check()
    yr, ar = oracle.gemm(blob, n, k, qs, ds, t_idx=np.arange(t))
    _assert_exact(host(y), yr, ar, f"prepared {n}x{k} t={t}")


def test_one_prepared_matrix_serves_every_token_count(q8):
    """The prepared form depends on (n, k) only: one buffer, several t (split
    and unsplit grids), interleaved with calls that take the other paths."""
    import torch

    n, k = 1536, 2048
    blob = syn.q8_0_weights(syn.rng(97, n, k), n, k)[0]
    w = dev(blob)
    wprep = q8.q8_0_gemm_prepare_weights(w, n, k)
    for i, t in enumerate((65, 16, 192, 40, 777, 1)):
        qs, ds = _plane(10 + i, t, k)
        qd, dd = dev(qs), dev(ds.view(np.int32))
        y_plain, y_prep = nan_f32(t, n), nan_f32(t, n)
        q8.q8_0_gemm(w, n, k, qd, dd, t, y_plain)
        q8.q8_0_gemm_prepared(w, wprep, n, k, qd, dd, t, y_prep)
        q8.q8_check()
        assert torch.equal(y_plain, y_prep), f"t={t}"


@pytest.mark.parametrize("t", [1, 9, 40])
def test_prepared_small_token_counts_read_the_q8_0_weights(q8, t):
    """t <= 64 takes the GEMV kernels on the Q8_0 matrix; no prepared form or
    workspace is needed (both may be absent)."""
    import torch

    n, k = 700, 1024
    blob = syn.q8_0_weights(syn.rng(98, n, k), n, k)[0]
    qs, ds = _plane(20, t, k)
    w, qd, dd = dev(blob), dev(qs), dev(ds.view(np.int32))
    assert q8.q8_0_gemm_prepared_workspace_bytes(n, t, k) == 0
    y_plain, y_prep = nan_f32(t, n), nan_f32(t, n)
    q8.q8_0_gemm(w, n, k, qd, dd, t, y_plain)
    q8.q8_0_gemm_prepared(w, None, n, k, qd, dd, t, y_prep)
    q8.q8_check()
    assert torch.equal(y_plain, y_prep)


def test_prepared_generic_shape_reads_the_q8_0_weights(q8):
    """(k/32) % 8 != 0 has no prepared form: the call runs the generic kernel on w."""
    import torch

    n, k, t = 300, 96, 100
    assert q8.q8_0_gemm_prepared_weights_bytes(n, k) == 0
    blob = syn.q8_0_weights(syn.rng(99, n, k), n, k)[0]
    qs, ds = _plane(30, t, k)
    w, qd, dd = dev(blob), dev(qs), dev(ds.view(np.int32))
    y_plain, y_prep = nan_f32(t, n), nan_f32(t, n)
    q8.q8_0_gemm(w, n, k, qd, dd, t, y_plain)
    q8.q8_0_gemm_prepared(w, None, n, k, qd, dd, t, y_prep)
    q8.q8_check()
    assert torch.equal(y_plain, y_prep)
    with pytest.raises(ValueError):
        q8.q8_0_gemm_prepare_weights(w, n, k)


def test_prepared_tc_path_without_prepared_weights_is_an_argument_error(q8):
    n, k, t = 256, 1024, 100
    qs, ds = _plane(40, t, k)
    y = nan_f32(t, n)
    with pytest.raises(q8.Q8Error) as e:
        q8.q8_0_gemm_prepared(None, None, n, k, dev(qs), dev(ds.view(np.int32)), t, y)
    assert e.value.status == 1  # Q8_ERR_ARG, before any device work


@pytest.mark.parametrize("n,k,t", [(18944, 3584, 3325), (3584, 18944, 3325)])
def test_prepared_full_size_prefill_shapes(q8, n, k, t):
    """The prefill chain's GEMM shapes as the bench times them: equal to
    q8_0_gemm bit for bit, no unwritten output, a sample against the oracle."""
    import torch

    blob = syn.q8_0_weights(syn.rng(100, n, k), n, k)[0]
    qs, ds = _plane(50, t, k)
    w, qd, dd = dev(blob), dev(qs), dev(ds.view(np.int32))
    wprep = q8.q8_0_gemm_prepare_weights(w, n, k)
    y_plain, y_prep = nan_f32(t, n), nan_f32(t, n)
    q8.q8_0_gemm(w, n, k, qd, dd, t, y_plain)
    q8.q8_0_gemm_prepared(None, wprep, n, k, qd, dd, t, y_prep)
    q8.q8_check()
    assert not torch.isnan(y_prep).any().item(), "unwritten outputs"
    assert torch.equal(y_plain, y_prep)
    g = syn.rng(101, n, k, t)
    ti = np.unique(np.concatenate([[0, t - 1], g.integers(0, t, 16)]))
    ni = np.unique(np.concatenate([[0, n - 1], g.integers(0, n, 64)]))
    yr, ar = oracle.gemm(blob, n, k, qs, ds, t_idx=ti, n_idx=ni)
    assert_gemm_close(host(y_prep)[np.ix_(ti, ni)], yr, ar, f"prepared {n}x{k} t={t} (sampled)")
