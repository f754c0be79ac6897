"""Build libq8proj.so in-tree with nvcc for sm_103a (GB300).

Each .cu file under csrc/ is compiled in parallel to an object file, then all
are linked into ``int8_quantized_projection_gb300/_build/libq8proj.so``
(static CUDA runtime).  ``python -m int8_quantized_projection_gb300.build``
builds it; ``--ptxas-v`` prints register/shared-memory usage per kernel.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libq8proj.so")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
           "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")] + [
        os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]


def _compile(src: str, ptxas_v: bool, extra: list[str], objdir: str = BUILD) -> tuple[str, str]:
    obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVFLAGS, *extra, "-c", src, "-o", obj]
    if ptxas_v:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, ptxas_v: bool = False, extra: list[str] | None = None, verbose: bool = False,
          lib_path: str | None = None) -> str:
    """Compile and link; skipped when the library is newer than every source.

    ``lib_path`` builds a separate copy there (with its objects beside it),
    always from scratch, e.g. with ``extra`` macro definitions; the in-tree
    library is left alone."""
    out = lib_path or LIB
    objdir = os.path.join(os.path.dirname(out), "obj") if lib_path else BUILD
    os.makedirs(objdir, exist_ok=True)
    extra = list(extra or [])
    if lib_path is None and not force and not ptxas_v and not extra and os.path.exists(LIB):
        newest = max(os.path.getmtime(p) for p in _deps())
        if os.path.getmtime(LIB) >= newest:
            return LIB
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, ptxas_v, extra, objdir), srcs))
    if verbose or ptxas_v:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = out + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True, ptxas_v="--ptxas-v" in sys.argv, verbose=True))
