"""q8_0_gemm_noalloc: the GEMM for callers that cannot allocate device memory at
the call (an engine that reserved all GPU memory for its own pool, a plugin
whose host forbids allocation after start-up, a latency-critical path that
cannot take cudaMalloc's implicit synchronisation).  Its scratch is a fixed
array inside the library, so these tests check that two calls in a row --
which reuse that array -- each give the same result as q8_0_gemm with a
caller-provided workspace, within the GEMM tolerance of the other tests, and
that a request larger than the array is refused.

This file is named so that pytest collects it last; it also passes when run
alone in a fresh process (the array's device address is looked up on the
first call on each device).
"""
import ctypes

import numpy as np
import pytest

import oracle
from int8_quantized_projection_gb300 import synthetic as syn

from ._parity import assert_gemm_close, dev, host, nan_f32

pytestmark = pytest.mark.gpu


def _case(seed, n, k, t):
    g = syn.rng(70, seed, n, k, t)
    blob = syn.q8_0_weights(g, n, k)[0]
    qs, ds = oracle.quantize(syn.activations(g, t, k, sigma=1.5, outlier_frac=0.01), ((t + 127) // 128) * 128)
    return blob, qs, ds


def _call_c_abi(q8, fn, blob_d, n, k, qs_d, ds_d, t, y):
    """Call an entry point through the C ABI with raw device pointers."""
    import torch

    lib = q8.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = [ctypes.c_void_p(blob_d.data_ptr()), n, k, ctypes.c_void_p(qs_d.data_ptr()),
            ctypes.c_void_p(ds_d.data_ptr()), t, qs_d.shape[0], ctypes.c_void_p(y.data_ptr())]
    if fn == "q8_0_gemm":
        ws = q8.gemm_workspace(n, t, k)
        args += [ctypes.c_void_p(ws.data_ptr()) if ws is not None else ctypes.c_void_p(0),
                 ws.numel() if ws is not None else 0]
        keep = ws
    else:
        keep = None
    st = getattr(lib, fn)(*args, stream)
    assert st == 0, f"{fn} returned {st}"
    assert lib.q8_check(stream) == 0
    del keep


def test_noalloc_gemm_two_calls_match_workspace_gemm(q8):
    import torch

    # two calls in a row with different shapes: the second reuses (and must
    # fully rewrite) the scratch the first one left behind
    for seed, (n, k, t) in enumerate([(1000, 3584, 300), (384, 2048, 129)]):
        blob, qs, ds = _case(seed, n, k, t)
        bd, qd, dd = dev(blob), dev(qs), dev(ds.view(np.int32))
        y_ref_gpu = nan_f32(t, n)
        _call_c_abi(q8, "q8_0_gemm", bd, n, k, qd, dd, t, y_ref_gpu)
        y = nan_f32(t, n)
        _call_c_abi(q8, "q8_0_gemm_noalloc", bd, n, k, qd, dd, t, y)
        assert torch.equal(y, y_ref_gpu), "no-allocation GEMM differs from the workspace GEMM"
        yr, ar = oracle.gemm(blob, n, k, qs, ds, t_idx=np.arange(t))
        assert_gemm_close(host(y), yr, ar, f"noalloc gemm {n}x{k} t={t}")


def test_noalloc_gemm_refuses_requests_beyond_its_scratch(q8):
    import torch

    lib = q8.lib()
    cap = lib.q8_0_gemm_noalloc_max_bytes()
    assert cap == 32 << 20
    t, k = 3325, 18944  # needs ~157 MB of scratch
    assert lib.q8_0_gemm_workspace_bytes(8, t, k) > cap
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    p = ctypes.c_void_p(dummy.data_ptr())
    st = lib.q8_0_gemm_noalloc(p, 8, k, p, p, t, t, p, ctypes.c_void_p(0))
    assert st == 7  # Q8_ERR_TOO_BIG, nothing enqueued
    assert b"scratch" in lib.q8_strerror(st)
