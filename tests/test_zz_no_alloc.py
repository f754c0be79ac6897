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


def test_noalloc_gemm_unsplit_and_near_its_limit(q8):
    """Two more shapes on the fixed scratch: one whose tiles fill the GPU (the
    GEMM runs without a k split and the weight pre-pass takes its wide form),
    and one whose scratch need is just under the array's size."""
    import torch

    lib = q8.lib()
    cap = lib.q8_0_gemm_noalloc_max_bytes()
    n, k = 4096, 2048
    t_hi = 65
    while lib.q8_0_gemm_workspace_bytes(n, t_hi + 64, k) <= cap:
        t_hi += 64
    assert cap - lib.q8_0_gemm_workspace_bytes(n, t_hi, k) < 64 * k * 2 + (1 << 20)
    for seed, (n_, k_, t_) in enumerate([(4096, 1024, 1920), (n, k, t_hi)]):
        assert lib.q8_0_gemm_workspace_bytes(n_, t_, k_) <= cap
        blob, qs, ds = _case(10 + seed, n_, k_, t_)
        bd, qd, dd = dev(blob), dev(qs), dev(ds.view(np.int32))
        y_ref_gpu = nan_f32(t_, n_)
        _call_c_abi(q8, "q8_0_gemm", bd, n_, k_, qd, dd, t_, y_ref_gpu)
        y = nan_f32(t_, n_)
        _call_c_abi(q8, "q8_0_gemm_noalloc", bd, n_, k_, qd, dd, t_, y)
        assert torch.equal(y, y_ref_gpu), f"no-allocation GEMM differs from the workspace GEMM at {n_}x{k_} t={t_}"
        g = syn.rng(71, seed)
        ti = np.unique(np.concatenate([[0, t_ - 1], g.integers(0, t_, 16)]))
        ni = np.unique(np.concatenate([[0, n_ - 1], g.integers(0, n_, 64)]))
        yr, ar = oracle.gemm(blob, n_, k_, qs, ds, t_idx=ti, n_idx=ni)
        assert_gemm_close(host(y)[np.ix_(ti, ni)], yr, ar, f"noalloc gemm {n_}x{k_} t={t_} (sampled)")


def test_noalloc_binding_refuses_bind_before_an_eager_call(q8):
    """The binding's bound (graph-capture) form needs the scratch address looked
    up by an earlier eager call on the device."""
    import torch

    saved = set(q8._binding._noalloc_devices)
    try:
        q8._binding._noalloc_devices.clear()
        n, k, t = 256, 256, 100
        w = torch.zeros(n * (k // 32) * 34, dtype=torch.uint8, device="cuda")
        qs, ds = q8.empty_plane(128, k)
        y = torch.empty(t, n, device="cuda")
        with pytest.raises(RuntimeError):
            q8.q8_0_gemm_noalloc(w, n, k, qs, ds, t, y, bind=True)
        qs.zero_(), ds.zero_()
        q8.q8_0_gemm_noalloc(w, n, k, qs, ds, t, y)
        q8.q8_check()
        q8.q8_0_gemm_noalloc(w, n, k, qs, ds, t, y, bind=True)()
        q8.q8_check()
        assert not torch.isnan(y).any() and not y.any()
    finally:
        q8._binding._noalloc_devices.update(saved)


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
