"""Bounded on-device waits: a wait that runs out is reported, never hangs.

Every kernel that waits on a barrier (the staged and small-batch GEMVs, the
tcgen05 GEMM, the many-row RMSNorm's row ring) gives up after a time limit, records Q8_ERR_DEVICE_TIMEOUT in
the library's error word and returns, after letting its own copies and
tensor-core work in flight land (those drain waits have a separate, long
limit).  q8_check reports the error and clears it.  The pages' counterpart is
the status a call returns instead of a wrong result ("54 - r51 -
producer-fused A-quantize mode 1", sec. 3.1: an allocation failure is
returned to the caller, which falls back).

The test builds a second copy of the library whose main-loop waits give up
at once (a zero limit: any wait that is not already satisfied times out;
drains keep their limit), loads it in a subprocess bounded by a host-side
timeout, and checks that a GEMM, a batch-1 GEMV, the small-batch GEMV on
both of its MMA paths and a many-row RMSNorm each report the timeout, that the report is cleared, and that nothing hangs.  A fresh process with the
normal library then gives a correct result.  Nothing here faults or hangs the
GPU: each wait is bounded, and every kernel reaches its exit after a timeout.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = textwrap.dedent(
    """
    import ctypes, sys
    sys.path.insert(0, ROOT)
    import numpy as np, torch
    from int8_quantized_projection_gb300 import _binding as bd, synthetic as syn
    lib = ctypes.CDLL(LIB)
    for name, (res, args) in bd.SIGNATURES.items():
        f = getattr(lib, name); f.restype = res; f.argtypes = args
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    out = {}
    # GEMM on the tcgen05 kernel (t > 64): its epilogue waits for the first
    # accumulator before any MMA can have finished
    n, k, t = 1024, 2048, 512
    w = torch.from_numpy(syn.q8_0_weights(syn.rng(75, 0), n, k)[0]).cuda()
    qs = torch.randint(-127, 128, (t, k), dtype=torch.int8, device="cuda")
    ds = torch.full((t, k // 32), 0x3C00, dtype=torch.int32, device="cuda")
    y = torch.empty(t, n, device="cuda")
    wsb = lib.q8_0_gemm_workspace_bytes(n, t, k)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    assert lib.q8_0_gemm(P(w), n, k, P(qs), P(ds), t, t, P(y), P(ws), wsb, st) == 0
    out["gemm"] = lib.q8_check(st)
    out["gemm_after"] = lib.q8_check(st)
    # batch-1 GEMV on the staged kernel: 93 MB of weights through per-warp rings
    n, k = 12288, 7168
    w = torch.from_numpy(syn.q8_0_weights(syn.rng(75, 1), n, k)[0]).cuda()
    qs = torch.randint(-127, 128, (1, k), dtype=torch.int8, device="cuda")
    ds = torch.full((1, k // 32), 0x3C00, dtype=torch.int32, device="cuda")
    y = torch.empty(n, device="cuda")
    assert lib.q8_0_gemv(P(w), n, k, P(qs), P(ds), P(y), st) == 0
    out["gemv"] = lib.q8_check(st)
    out["gemv_after"] = lib.q8_check(st)
    # small-batch GEMV: t = 16 (f16 path, where the consumer warps agree on each
    # stage's arrival at a barrier and leave together) and t = 4 (int8 path)
    n, k = 4096, 7168
    w = torch.from_numpy(syn.q8_0_weights(syn.rng(75, 2), n, k)[0]).cuda()
    qs = torch.randint(-127, 128, (128, k), dtype=torch.int8, device="cuda")
    ds = torch.full((128, k // 32), 0x3C00, dtype=torch.int32, device="cuda")
    for tt in (16, 4):
        y = torch.empty(tt, n, device="cuda")
        assert lib.q8_0_gemv_batched(P(w), n, k, P(qs), P(ds), tt, P(y), st) == 0
        out["small%d" % tt] = lib.q8_check(st)
        out["small%d_after" % tt] = lib.q8_check(st)
    # RMSNorm over many rows: the shared-memory row ring waits for each row's copy
    rows, d = 3325, 3584
    x = torch.randn(rows, d, device="cuda")
    nw = torch.ones(d, device="cuda")
    qs = torch.empty(3328, d, dtype=torch.int8, device="cuda")
    ds = torch.empty(3328, d // 32, dtype=torch.int32, device="cuda")
    assert lib.rmsnorm_quant(P(x), P(nw), ctypes.c_float(1e-6), None, rows, d, P(qs), P(ds), 3328, st) == 0
    out["rmsnorm"] = lib.q8_check(st)
    out["rmsnorm_after"] = lib.q8_check(st)
    print("RESULT", out)
    """
)

_FRESH = textwrap.dedent(
    """
    import sys
    sys.path.insert(0, ROOT)
    import numpy as np, torch
    import oracle
    import int8_quantized_projection_gb300 as q8
    from int8_quantized_projection_gb300 import synthetic as syn
    n, k, t = 1024, 2048, 512
    g = syn.rng(76, 0)
    blob = syn.q8_0_weights(g, n, k)[0]
    qs, ds = oracle.quantize(syn.activations(g, t, k), t)
    y = torch.full((t, n), float("nan"), device="cuda")
    q8.q8_0_gemm(torch.from_numpy(blob).cuda(), n, k, torch.from_numpy(qs).cuda(),
                 torch.from_numpy(ds.view(np.int32)).cuda(), t, y)
    q8.q8_check()
    yr, ar = oracle.gemm(blob, n, k, qs, ds)
    err = float(np.max(np.abs(y.cpu().numpy().astype(np.float64) - yr) / np.maximum(ar, 1e-300)))
    print("RESULT", err)
    """
)


def _run(code, **env):
    prog = "".join(f"{k} = {v!r}\n" for k, v in env.items()) + code
    r = subprocess.run([sys.executable, "-c", prog], capture_output=True, text=True, timeout=180)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("RESULT")][-1]
    return eval(line.split(" ", 1)[1])  # a dict or float printed by the child


def test_waits_that_run_out_report_a_timeout(tmp_path):
    from int8_quantized_projection_gb300 import build

    lib = build.build(extra=["-DQ8_WAIT_LIMIT_NS=0ull"], lib_path=str(tmp_path / "libq8proj_waits0.so"))
    got = _run(_CHILD, ROOT=ROOT, LIB=lib)
    calls = ("gemm", "gemv", "small16", "small4", "rmsnorm")
    assert all(got[c] == 5 for c in calls), got  # Q8_ERR_DEVICE_TIMEOUT
    assert all(got[c + "_after"] == 0 for c in calls), got  # then cleared
    # a fresh process with the normal library computes correctly
    err = _run(_FRESH, ROOT=ROOT)
    assert err <= 1e-5
