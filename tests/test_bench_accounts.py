"""The bench's algorithmic byte and op counts (the numerators of every
roofline figure) against the bytes the path actually moves, measured from
the objects themselves: synthetic weight blobs, the oracle's plane rows and
f32 arrays.  The expected totals for the configured shapes are spelled out
as numbers, so a change to a formula or a format shows up here."""
import os
import sys

import numpy as np

import oracle
from int8_quantized_projection_gb300 import synthetic as syn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _row_bytes(blob_fn, k):
    """Bytes of one weight row in a format: a 2-row blob halved."""
    return blob_fn(syn.rng(95, k), 2, k)[0].nbytes // 2


def _plane_row_bytes(k):
    qs, ds = oracle.quantize(np.zeros((1, k), np.float32))
    return qs.nbytes + ds.nbytes


def _gemv_moved(n, k, blob_fn=syn.q8_0_weights):
    return n * _row_bytes(blob_fn, k) + _plane_row_bytes(k) + n * 4


def test_gemv_accounts():
    for n, k in bench.DECODE_SHAPES:
        assert bench.bytes_gemv(n, k) == _gemv_moved(n, k)
    assert bench.bytes_gemv(12288, 7168) == 93_642_624
    assert bench.bytes_q4a_gemv(12288, 7168) == _gemv_moved(12288, 7168, syn.q4a_weights)


def test_producer_accounts():
    T, d, nf = 3325, 3584, 18944
    f32 = np.dtype(np.float32).itemsize
    # rmsnorm: x read, w read, y written (mode 1), the plane rows written
    assert bench.bytes_rmsnorm_quant(T, d) == 2 * T * d * f32 + d * f32 + T * _plane_row_bytes(d) == 108_755_136
    assert bench.bytes_rmsnorm_quant(T, d, False) == bench.bytes_rmsnorm_quant(T, d) - T * d * f32
    # swiglu: gate and up read, y written (mode 1), the plane rows written
    assert bench.bytes_swiglu_quant(T, nf) == 3 * T * nf * f32 + T * _plane_row_bytes(nf) == 826_728_000
    assert bench.bytes_swiglu_quant(T, nf, False) == bench.bytes_swiglu_quant(T, nf) - T * nf * f32
    assert bench.bytes_quantize(1, 7168) == 7168 * f32 + _plane_row_bytes(7168)


def test_gemm_ops():
    assert bench.ops_gemm(3325, 18944, 3584) == 2 * 3325 * 18944 * 3584  # 451.5 G int8 ops


def test_grouped_and_layer_stack_accounts():
    k, ns = bench.SHARED["d"], bench.SHARED["ns"]
    # one activation read for the whole group
    assert bench.bytes_gemv_group(k, ns) == sum(n * _row_bytes(syn.q8_0_weights, k) + 4 * n for n in ns) \
        + _plane_row_bytes(k)
    L = bench.LAYERS
    w = sum(n * _row_bytes(syn.q8_0_weights, kk) for kk, group in bench.layer_groups() for n in group)
    head = L["vocab"] * _row_bytes(syn.q8_0_weights, L["d"])
    assert L["layers"] * w + head == 7_512_178_688  # every projection of the stack and the LM head
    assert 7_512_178_688 < bench.bytes_layer_stack() < 7_512_178_688 * 1.003  # + activations, planes, outputs


def test_fused_accounts():
    """A fused launch moves the weights, the outputs and the producer's f32
    inputs once; no plane is written or read."""
    f32 = np.dtype(np.float32).itemsize
    k, ns = bench.SHARED["d"], bench.SHARED["ns"]
    weights_out = sum(n * _row_bytes(syn.q8_0_weights, k) + 4 * n for n in ns)
    assert bench.bytes_gemv_fused(k, ns, "rmsnorm") == weights_out + 2 * k * f32   # x and the norm weight
    assert bench.bytes_gemv_fused(k, ns, "quant") == weights_out + k * f32
    assert bench.bytes_gemv_fused(k, ns, "swiglu") == weights_out + 2 * k * f32    # gate and up
    assert bench.bytes_shared(fused=True) == bench.bytes_shared() - bench.bytes_rmsnorm_quant(1, k, False) \
        - _plane_row_bytes(k) + 2 * k * f32
    L = bench.LAYERS
    d, nf = L["d"], L["nf"]
    # per layer: 2 RMSNorm inputs (x, w), the attention output, gate + up; the final norm's x and w
    inputs = L["layers"] * (2 * 2 * d + d + 2 * nf) * f32 + 2 * d * f32
    outputs = (L["layers"] * sum(n for _, group in bench.layer_groups() for n in group) + L["vocab"]) * f32
    every = ("qkv", "o", "gu", "down", "head")
    assert bench.bytes_layer_stack(every) == 7_512_178_688 + inputs + outputs
    # fusing one producer removes its plane write and read and its mode-2 bytes, adds nothing else
    one = bench.bytes_layer_stack() - bench.bytes_layer_stack(("qkv",))
    assert one == L["layers"] * (bench.bytes_rmsnorm_quant(1, d, False) + _plane_row_bytes(d) - 2 * d * f32)


def test_fused_decode_accounts():
    """The decode step with its k = 7168 quantize inside the grouped GEMV: the plane's write and its reads by the two
    projections (counted per projection in the unfused step) are gone, the f32 activation is read once."""
    assert bench.decode_bytes() - bench.decode_bytes(fused=True) == 3 * _plane_row_bytes(7168)


def test_gate_up_pair_accounts():
    """Gate/up writing the SwiGLU plane in its epilogue: per layer the gate/up f32 outputs (written, then read by
    swiglu_quant) disappear; every other byte stays."""
    f32 = np.dtype(np.float32).itemsize
    L = bench.LAYERS
    nf = L["nf"]
    assert bench.bytes_layer_stack() - bench.bytes_layer_stack(("gu_pair",)) == L["layers"] * 4 * nf * f32
