"""Host-side checks of the C ABI: the library builds, loads without a GPU, exports
every symbol include/q8proj.h declares, and rejects bad arguments before it
touches the device (no compute call is made here)."""
import ctypes
import os
import re

import pytest

import int8_quantized_projection_gb300 as q8p
from int8_quantized_projection_gb300 import _binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q8proj.h")

FAKE = 0x10000      # 16-byte aligned, never dereferenced: every call below fails validation first
MISALIGNED = 0x10004


@pytest.fixture(scope="module")
def lib():
    build.build()
    return q8p.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^Q8_API\s+[\w\s\*]+?\**\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_abi():
    assert declared_symbols() == sorted(_binding.SIGNATURES)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    # and nothing else of ours leaks (kernels and helpers are hidden)
    out = os.popen(f"nm -D --defined-only {build.LIB}").read().split("\n")
    ours = {ln.split()[-1] for ln in out if ln.strip() and ln.split()[-1].startswith(("q8", "q4a", "quantize", "rmsnorm",
                                                                                       "swiglu"))}
    assert ours == set(declared_symbols())


def test_plane_rows_and_strerror(lib):
    assert lib.q8_plane_rows(1) == 128
    assert lib.q8_plane_rows(128) == 128
    assert lib.q8_plane_rows(3325) == 3328
    assert lib.q8_plane_rows(0) == 128
    for st in range(0, 7):
        assert lib.q8_strerror(st)
    assert lib.q8_strerror(99) == b"unknown status"


P = ctypes.c_void_p


def test_argument_errors_are_reported_before_any_device_work(lib):
    s = P(0)
    ERR_ARG, ERR_ALIGN = 1, 2
    # quantize_q8_0: k % 32, rows_pad < rows, null plane
    assert lib.quantize_q8_0(P(FAKE), 4, 48, P(FAKE), P(FAKE), 4, s) == ERR_ARG
    assert lib.quantize_q8_0(P(FAKE), 4, 64, P(FAKE), P(FAKE), 3, s) == ERR_ARG
    assert lib.quantize_q8_0(P(FAKE), 4, 64, P(0), P(FAKE), 4, s) == ERR_ARG
    assert lib.quantize_q8_0(P(0), 4, 64, P(FAKE), P(FAKE), 4, s) == ERR_ARG
    assert lib.quantize_q8_0(P(FAKE), 4, 64, P(MISALIGNED), P(FAKE), 4, s) == ERR_ALIGN
    assert lib.quantize_q8_0(P(MISALIGNED), 4, 64, P(FAKE), P(FAKE), 4, s) == ERR_ALIGN
    # rmsnorm_quant: d limit and alignment
    assert lib.rmsnorm_quant(P(FAKE), P(FAKE), 1e-6, P(FAKE), 2, 32768 + 32, P(FAKE), P(FAKE), 2, s) == ERR_ARG
    assert lib.rmsnorm_quant(P(FAKE), P(MISALIGNED), 1e-6, P(FAKE), 2, 64, P(FAKE), P(FAKE), 2, s) == ERR_ALIGN
    # swiglu_quant
    assert lib.swiglu_quant(P(FAKE), P(FAKE), P(FAKE), 2, 40, P(FAKE), P(FAKE), 2, s) == ERR_ARG
    assert lib.swiglu_quant(P(FAKE), P(FAKE), P(MISALIGNED), 2, 64, P(FAKE), P(FAKE), 2, s) == ERR_ALIGN
    # q8_0_gemv
    assert lib.q8_0_gemv(P(FAKE), 0, 64, P(FAKE), P(FAKE), P(FAKE), s) == ERR_ARG
    assert lib.q8_0_gemv(P(FAKE), 8, 100, P(FAKE), P(FAKE), P(FAKE), s) == ERR_ARG
    assert lib.q8_0_gemv(P(FAKE + 2), 8, 64, P(FAKE), P(FAKE), P(FAKE), s) == ERR_ALIGN
    # q8_0_gemm: rows_pad < t, t < 1, workspace missing or too small
    ws = lib.q8_0_gemm_workspace_bytes(8, 100, 256)
    up = lambda v: -(-v // 1024) * 1024
    # f16 weights | f16 activation | d_w per 128-row tile | d_a per 192-token tile, each from a 1 KiB boundary
    assert ws == up(up(up(8 * 256 * 2) + 100 * 256 * 2) + 1 * 8 * 128 * 4) + up(1 * 8 * 192 * 4)
    # a grid of 2 tiles splits k 8 ways (32 stages of 2 blocks, at least 4 per split): + 8 x t x n f32 partial tiles
    ws2 = lib.q8_0_gemm_workspace_bytes(256, 130, 2048)
    assert ws2 == up(up(up(up(256 * 2048 * 2) + 130 * 2048 * 2) + 2 * 64 * 128 * 4) + 1 * 64 * 192 * 4) \
        + 8 * 130 * 256 * 4
    assert lib.q8_0_gemm_workspace_bytes(18944, 3325, 3584) == up(up(up(up(18944 * 3584 * 2) + 3325 * 3584 * 2)
                                                                     + 148 * 112 * 128 * 4) + 18 * 112 * 192 * 4)
    # 4 x 3 = 12 tiles: k split 12 ways (152 // 12 = 12, the cap; 56 stages allow 14) -> 12 x t x n partials
    assert lib.q8_0_gemm_workspace_bytes(512, 512, 3584) == up(up(up(up(512 * 3584 * 2) + 512 * 3584 * 2)
                                                                 + 4 * 112 * 128 * 4) + 3 * 112 * 192 * 4) \
        + 12 * 512 * 512 * 4
    # 4 x 11 = 44 tiles: 152 // 44 = 3 splits
    assert lib.q8_0_gemm_workspace_bytes(512, 2048, 3584) == up(up(up(up(512 * 3584 * 2) + 2048 * 3584 * 2)
                                                                  + 4 * 112 * 128 * 4) + 11 * 112 * 192 * 4) \
        + 3 * 2048 * 512 * 4
    # many tiles whose last wave would leave most SMs idle: 28 x 18 = 504 tiles fill 3.3 waves of 152 CTAs, so
    # k (296 stages) is split 3 ways (9.9 waves) -> 3 x t x n f32 partial tiles; gate/up's 2664 tiles stay unsplit
    assert lib.q8_0_gemm_workspace_bytes(3584, 3325, 18944) == up(up(up(up(3584 * 18944 * 2) + 3325 * 18944 * 2)
                                                                    + 28 * 592 * 128 * 4) + 18 * 592 * 192 * 4) \
        + 3 * 3325 * 3584 * 4
    assert lib.q8_0_gemm_workspace_bytes(8, 20, 64) == 0      # k/32 % 8 != 0: generic kernel, no workspace
    assert lib.q8_0_gemm_workspace_bytes(8, 16, 256) == 0     # t <= 16: small-batch kernel, no workspace
    assert lib.q8_0_gemm_workspace_bytes(8, 64, 256) == 0     # t <= 64: 16-token slices, no workspace
    assert lib.q8_0_gemm_workspace_bytes(8, 65, 256) > 0      # the GEMM from 65 tokens
    assert lib.q8_0_gemm(P(FAKE), 8, 64, P(FAKE), P(FAKE), 5, 4, P(FAKE), P(0), 0, s) == ERR_ARG
    assert lib.q8_0_gemm(P(FAKE), 8, 64, P(FAKE), P(FAKE), 0, 4, P(FAKE), P(0), 0, s) == ERR_ARG
    assert lib.q8_0_gemm(P(FAKE), 8, 256, P(FAKE), P(FAKE), 100, 100, P(FAKE), P(0), ws, s) == ERR_ARG
    assert lib.q8_0_gemm(P(FAKE), 8, 256, P(FAKE), P(FAKE), 100, 100, P(FAKE), P(FAKE), ws - 1, s) == ERR_ARG
    assert lib.q8_0_gemm(P(FAKE), 8, 256, P(FAKE), P(FAKE), 100, 100, P(FAKE), P(MISALIGNED), ws, s) == ERR_ALIGN
    assert lib.q8_0_gemm(P(FAKE), 8, 64, P(FAKE), P(MISALIGNED), 4, 4, P(FAKE), P(0), 0, s) == ERR_ALIGN
    # q8_0_gemv_batched: tokens outside 1..16, k % 32, alignment
    assert lib.q8_0_gemv_batched(P(FAKE), 8, 256, P(FAKE), P(FAKE), 0, P(FAKE), s) == ERR_ARG
    assert lib.q8_0_gemv_batched(P(FAKE), 8, 256, P(FAKE), P(FAKE), 17, P(FAKE), s) == ERR_ARG
    assert lib.q8_0_gemv_batched(P(FAKE), 8, 100, P(FAKE), P(FAKE), 4, P(FAKE), s) == ERR_ARG
    assert lib.q8_0_gemv_batched(P(FAKE), 8, 256, P(FAKE), P(FAKE), 4, P(MISALIGNED), s) == ERR_ALIGN
    # q8_0_gemv_batched_grouped: count 1..8, tokens 1..16, k % 32, each projection's pointers and n, alignment
    grp = (_binding.GemvProj * 2)(_binding.GemvProj(FAKE, 8, FAKE), _binding.GemvProj(FAKE, 40, FAKE))
    gp = ctypes.cast(grp, ctypes.c_void_p)
    bgrp = lib.q8_0_gemv_batched_grouped
    assert bgrp(None, 1, 256, P(FAKE), P(FAKE), 4, s) == ERR_ARG
    assert bgrp(gp, 0, 256, P(FAKE), P(FAKE), 4, s) == ERR_ARG
    assert bgrp(gp, 9, 256, P(FAKE), P(FAKE), 4, s) == ERR_ARG
    assert bgrp(gp, 2, 256, P(FAKE), P(FAKE), 0, s) == ERR_ARG
    assert bgrp(gp, 2, 256, P(FAKE), P(FAKE), 17, s) == ERR_ARG
    assert bgrp(gp, 2, 100, P(FAKE), P(FAKE), 4, s) == ERR_ARG
    assert bgrp(gp, 2, 256, P(0), P(FAKE), 4, s) == ERR_ARG
    assert bgrp(gp, 2, 256, P(FAKE), P(MISALIGNED), 4, s) == ERR_ALIGN
    grp[1] = _binding.GemvProj(FAKE, 0, FAKE)
    assert bgrp(gp, 2, 256, P(FAKE), P(FAKE), 4, s) == ERR_ARG
    grp[1] = _binding.GemvProj(FAKE, 40, None)
    assert bgrp(gp, 2, 256, P(FAKE), P(FAKE), 4, s) == ERR_ARG
    grp[1] = _binding.GemvProj(FAKE, 40, MISALIGNED)
    assert bgrp(gp, 2, 256, P(FAKE), P(FAKE), 4, s) == ERR_ALIGN
    # q4a_gemv: k % 128, n < 1, alignment
    assert lib.q4a_gemv(P(FAKE), 8, 96, P(FAKE), P(FAKE), P(FAKE), s) == ERR_ARG
    assert lib.q4a_gemv(P(FAKE), 0, 256, P(FAKE), P(FAKE), P(FAKE), s) == ERR_ARG
    assert lib.q4a_gemv(P(FAKE + 4), 8, 256, P(FAKE), P(FAKE), P(FAKE), s) == ERR_ALIGN
    # q4a_gemv_batched: k % 256 (whole 8-block pieces), tokens 1..16, alignment
    assert lib.q4a_gemv_batched(P(FAKE), 8, 128, P(FAKE), P(FAKE), 4, P(FAKE), s) == ERR_ARG
    assert lib.q4a_gemv_batched(P(FAKE), 8, 256, P(FAKE), P(FAKE), 0, P(FAKE), s) == ERR_ARG
    assert lib.q4a_gemv_batched(P(FAKE), 8, 256, P(FAKE), P(FAKE), 17, P(FAKE), s) == ERR_ARG
    assert lib.q4a_gemv_batched(P(0), 8, 256, P(FAKE), P(FAKE), 4, P(FAKE), s) == ERR_ARG
    assert lib.q4a_gemv_batched(P(FAKE), 8, 256, P(FAKE), P(FAKE), 4, P(MISALIGNED), s) == ERR_ALIGN
    # q4a_gemv_batched_grouped: count 1..8, k % 256, tokens 1..16, descriptors, alignment
    qgrp = (_binding.GemvProj * 2)(_binding.GemvProj(FAKE, 8, FAKE), _binding.GemvProj(FAKE, 40, FAKE))
    qp = ctypes.cast(qgrp, ctypes.c_void_p)
    qb = lib.q4a_gemv_batched_grouped
    assert qb(None, 1, 256, P(FAKE), P(FAKE), 4, s) == ERR_ARG
    assert qb(qp, 0, 256, P(FAKE), P(FAKE), 4, s) == ERR_ARG
    assert qb(qp, 9, 256, P(FAKE), P(FAKE), 4, s) == ERR_ARG
    assert qb(qp, 2, 128, P(FAKE), P(FAKE), 4, s) == ERR_ARG
    assert qb(qp, 2, 256, P(FAKE), P(FAKE), 0, s) == ERR_ARG
    assert qb(qp, 2, 256, P(FAKE), P(FAKE), 17, s) == ERR_ARG
    assert qb(qp, 2, 256, P(FAKE), P(MISALIGNED), 4, s) == ERR_ALIGN
    qgrp[1] = _binding.GemvProj(FAKE, 0, FAKE)
    assert qb(qp, 2, 256, P(FAKE), P(FAKE), 4, s) == ERR_ARG
    qgrp[1] = _binding.GemvProj(MISALIGNED, 40, FAKE)
    assert qb(qp, 2, 256, P(FAKE), P(FAKE), 4, s) == ERR_ALIGN
    # q8_0_gemv_fused: producer code, its inputs, the staged path's k, RMSNorm's row limit, alignment
    one = (_binding.GemvProj * 1)(_binding.GemvProj(FAKE, 8, FAKE))
    pr = ctypes.cast(one, ctypes.c_void_p)
    fused = lib.q8_0_gemv_fused
    assert fused(pr, 1, 256, 0, P(FAKE), P(0), P(0), 0.0, s) == ERR_ARG           # no producer 0
    assert fused(pr, 1, 256, 4, P(FAKE), P(0), P(0), 0.0, s) == ERR_ARG           # nor 4
    assert fused(pr, 0, 256, 1, P(FAKE), P(0), P(0), 0.0, s) == ERR_ARG           # count 0
    assert fused(pr, 1, 256, 1, P(0), P(0), P(0), 0.0, s) == ERR_ARG              # x missing
    assert fused(pr, 1, 256, 3, P(FAKE), P(0), P(0), 0.0, s) == ERR_ARG           # up missing
    assert fused(pr, 1, 256, 2, P(FAKE), P(0), P(0), 1e-6, s) == ERR_ARG          # norm weight missing
    assert fused(pr, 1, 2080, 1, P(FAKE), P(0), P(0), 0.0, s) == ERR_ARG          # 65 blocks per row
    assert fused(pr, 1, 65536 + 256, 1, P(FAKE), P(0), P(0), 0.0, s) == ERR_ARG   # row longer than the staging
    assert fused(pr, 1, 32768 + 256, 2, P(FAKE), P(0), P(FAKE), 1e-6, s) == ERR_ARG  # RMSNorm limit
    assert fused(pr, 1, 256, 1, P(MISALIGNED), P(0), P(0), 0.0, s) == ERR_ALIGN
    assert fused(pr, 1, 256, 3, P(FAKE), P(MISALIGNED), P(0), 0.0, s) == ERR_ALIGN
    assert fused(pr, 1, 256, 2, P(FAKE), P(0), P(MISALIGNED), 1e-6, s) == ERR_ALIGN
    bad = (_binding.GemvProj * 1)(_binding.GemvProj(FAKE + 8, 8, FAKE))
    assert fused(ctypes.cast(bad, ctypes.c_void_p), 1, 256, 1, P(FAKE), P(0), P(0), 0.0, s) == ERR_ALIGN
    # q8_0_gemv_gate_up: nf % 32, k on the staged whole-row path (2048 < k <= 65536), producer and its inputs,
    # the output plane, alignment
    gu = lambda nf, k, qs, ds, prod, a, nw, yg, qo, do: lib.q8_0_gemv_gate_up(  # noqa: E731
        P(FAKE), P(FAKE), nf, k, P(qs), P(ds), prod, P(a), P(nw), 1e-6, P(yg), P(0), P(qo), P(do), s)
    assert gu(48, 3584, FAKE, FAKE, 0, 0, 0, 0, FAKE, FAKE) == ERR_ARG          # nf % 32
    assert gu(64, 2048, FAKE, FAKE, 0, 0, 0, 0, FAKE, FAKE) == ERR_ARG          # rows share a warp at k <= 2048
    assert gu(64, 2080, FAKE, FAKE, 0, 0, 0, 0, FAKE, FAKE) == ERR_ARG          # 65 blocks per row
    assert gu(64, 65536 + 256, FAKE, FAKE, 0, 0, 0, 0, FAKE, FAKE) == ERR_ARG   # longer than the staging
    assert gu(64, 3584, 0, FAKE, 0, 0, 0, 0, FAKE, FAKE) == ERR_ARG             # plane missing
    assert gu(64, 3584, 0, 0, 3, FAKE, 0, 0, FAKE, FAKE) == ERR_ARG             # no SwiGLU producer here
    assert gu(64, 3584, 0, 0, 2, FAKE, 0, 0, FAKE, FAKE) == ERR_ARG             # norm weight missing
    assert gu(64, 32768 + 256, 0, 0, 2, FAKE, FAKE, 0, FAKE, FAKE) == ERR_ARG   # RMSNorm limit
    assert gu(64, 3584, FAKE, FAKE, 0, 0, 0, 0, 0, FAKE) == ERR_ARG             # output plane missing
    assert gu(64, 3584, FAKE, FAKE, 0, 0, 0, 0, MISALIGNED, FAKE) == ERR_ALIGN
    assert gu(64, 3584, FAKE, FAKE, 0, 0, 0, MISALIGNED, FAKE, FAKE) == ERR_ALIGN
    assert gu(64, 3584, 0, 0, 1, MISALIGNED, 0, 0, FAKE, FAKE) == ERR_ALIGN


def test_prepared_gemm_sizes_and_argument_errors(lib):
    """The prepared-weight GEMM entry points: sizes as a function of the shape
    (the weight pre-pass's two parts; the workspace without them) and the
    argument errors reported before any device work."""
    s = P(0)
    ERR_ARG, ERR_ALIGN = 1, 2
    up = lambda v: -(-v // 1024) * 1024  # noqa: E731
    # [f16 codes n x k | d_w per 128-row tile], each from a 1 KiB boundary
    assert lib.q8_0_gemm_prepared_weights_bytes(8, 256) == up(up(8 * 256 * 2) + 1 * 8 * 128 * 4)
    assert lib.q8_0_gemm_prepared_weights_bytes(18944, 3584) == up(up(18944 * 3584 * 2) + 148 * 112 * 128 * 4)
    assert lib.q8_0_gemm_prepared_weights_bytes(8, 96) == 0           # (k/32) % 8 != 0: no tcgen05 path
    assert lib.q8_0_gemm_prepared_weights_bytes(65535 * 128 + 1, 256) == 0  # past the grid's weight-row tiles
    # the workspace is q8_0_gemm's without the weight parts
    assert lib.q8_0_gemm_prepared_workspace_bytes(8, 100, 256) == up(up(100 * 256 * 2) + 1 * 8 * 192 * 4)
    for n, t, k in ((18944, 3325, 3584), (256, 130, 2048), (512, 512, 3584)):
        full = lib.q8_0_gemm_workspace_bytes(n, t, k)
        prep = lib.q8_0_gemm_prepared_workspace_bytes(n, t, k)
        wparts = up(n * k * 2) + up(-(-n // 128) * (k // 32) * 128 * 4)
        assert prep == full - wparts, (n, t, k)
    assert lib.q8_0_gemm_prepared_workspace_bytes(8, 64, 256) == 0  # t <= 64: no workspace
    assert lib.q8_0_gemm_prepared_workspace_bytes(8, 100, 96) == 0  # generic kernel
    wpb = lib.q8_0_gemm_prepared_weights_bytes(8, 256)
    prep = lib.q8_0_gemm_prepare_weights
    assert prep(P(0), 8, 256, P(FAKE), wpb, s) == ERR_ARG               # no weights
    assert prep(P(FAKE), 8, 256, P(0), wpb, s) == ERR_ARG               # no buffer
    assert prep(P(FAKE), 8, 256, P(FAKE), wpb - 1, s) == ERR_ARG        # short buffer
    assert prep(P(FAKE), 8, 96, P(FAKE), 1 << 20, s) == ERR_ARG         # no prepared form
    assert prep(P(FAKE), 0, 256, P(FAKE), wpb, s) == ERR_ARG            # n < 1
    assert prep(P(FAKE + 2), 8, 256, P(FAKE), wpb, s) == ERR_ALIGN
    assert prep(P(FAKE), 8, 256, P(MISALIGNED), wpb, s) == ERR_ALIGN
    ws = lib.q8_0_gemm_prepared_workspace_bytes(8, 100, 256)
    gp = lambda w, wp, k, t, rp, wsp, wsb: lib.q8_0_gemm_prepared(  # noqa: E731
        P(w), P(wp), 8, k, P(FAKE), P(FAKE), t, rp, P(FAKE), P(wsp), wsb, s)
    assert gp(FAKE, 0, 256, 100, 100, FAKE, ws) == ERR_ARG          # the tcgen05 path needs the prepared weights
    assert gp(0, FAKE, 256, 40, 40, 0, 0) == ERR_ARG                # t <= 64 reads the Q8_0 weights
    assert gp(0, FAKE, 96, 100, 100, 0, 0) == ERR_ARG               # so does the generic kernel
    assert gp(0, FAKE, 256, 100, 100, FAKE, ws - 1) == ERR_ARG      # short workspace
    assert gp(0, FAKE, 256, 100, 100, 0, ws) == ERR_ARG             # no workspace
    assert gp(0, FAKE, 256, 100, 99, FAKE, ws) == ERR_ARG           # rows_pad < t
    assert gp(0, FAKE, 256, 0, 4, FAKE, ws) == ERR_ARG              # t < 1
    assert gp(0, MISALIGNED, 256, 100, 100, FAKE, ws) == ERR_ALIGN
    assert gp(0, FAKE, 256, 100, 100, MISALIGNED, ws) == ERR_ALIGN
    assert gp(FAKE + 2, 0, 256, 40, 40, 0, 0) == ERR_ALIGN


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _binding.lib()
