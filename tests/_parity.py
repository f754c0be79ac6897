"""Shared helpers of the GPU parity tests: moving seeded numpy inputs to the
device, poisoning outputs, and the comparison rules.

Comparison rules:
  * planes (qs bytes, d bits, int16 ssum): bit-exact against the oracle;
  * f32 producer outputs (RMSNorm, SwiGLU): |y - y_ref| <= 1e-5 |y_ref| + 2^-100,
    y_ref the oracle's fp64 value;
  * GEMV/GEMM outputs: |y - y_ref| <= 1e-5 * A, A = sum_b |d_w d_a isum_b|
    (the scale of the sum the kernel evaluates in a different order); where
    A = 0 the output must be exactly 0.
"""
import numpy as np

Y_RTOL = 1e-5
Y_ATOL = 2.0 ** -100
GEMM_TOL = 1e-5
POISON_BYTE = 0xA5


def dev(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.detach().cpu().numpy()


def poisoned_plane(rows_pad, k):
    import torch

    qs = torch.full((rows_pad, k), POISON_BYTE - 256, dtype=torch.int8, device="cuda")
    ds = torch.full((rows_pad, k // 32), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    return qs, ds


def nan_f32(*shape):
    import torch

    return torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")


def assert_plane_equal(qs_gpu, ds_gpu, qs_ref, ds_ref, what=""):
    qg = host(qs_gpu).view(np.int8)
    dg = host(ds_gpu).view(np.uint32)
    assert qg.shape == qs_ref.shape and dg.shape == ds_ref.shape
    bad_q = np.argwhere(qg != qs_ref)
    bad_d = np.argwhere(dg != ds_ref)
    assert bad_q.size == 0, f"{what}: {len(bad_q)} qs bytes differ, first at {bad_q[:4].tolist()}"
    assert bad_d.size == 0, f"{what}: {len(bad_d)} ds words differ, first at {bad_d[:4].tolist()}"


def assert_y_close(y_gpu, y_ref, what=""):
    yg = host(y_gpu).astype(np.float64)
    assert not np.isnan(yg).any(), f"{what}: unwritten (NaN) outputs"
    err = np.abs(yg - y_ref)
    lim = Y_RTOL * np.abs(y_ref) + Y_ATOL
    bad = np.argwhere(err > lim)
    assert bad.size == 0, f"{what}: {len(bad)} outputs beyond 1e-5, worst rel {np.max(err / np.maximum(np.abs(y_ref), 1e-300)):.3e}"


def gemm_errors(y_gpu, y_ref, absum):
    yg = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(yg - y_ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        rel_a = np.where(absum > 0, err / absum, np.where(err == 0, 0.0, np.inf))
    return err, rel_a


def assert_gemm_close(y_gpu, y_ref, absum, what=""):
    yg = np.asarray(y_gpu, dtype=np.float64)
    assert not np.isnan(yg).any(), f"{what}: {int(np.isnan(yg).sum())} unwritten (NaN) outputs"
    err, rel_a = gemm_errors(yg, y_ref, absum)
    worst = float(rel_a.max()) if rel_a.size else 0.0
    assert worst <= GEMM_TOL, f"{what}: max |dy|/A = {worst:.3e} > {GEMM_TOL}"
    return worst
