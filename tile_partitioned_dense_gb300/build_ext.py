"""Builds libtpgemm.so in-tree with nvcc for sm_103a.

Twelve translation units compiled in parallel: the host library
(tpgemm.cu), the streaming-kernel instantiations (stream_inst.cu), the
block-scaled kernel's MXFP8 ones (mx_inst.cu) and FP4 ones (fp4_inst.cu with
-DTPG_FP4=1 for NVFP4 and 2 for MXFP4), the tiled-kernel instantiations, one
per fused-epilogue mode (tiled_inst.cu with -DTPG_EPI=0..5, 5 being the plain
epilogue for alpha == 1), and the grouped tiled kernel (-DTPG_GROUPED=1);
then one link.
"""
from __future__ import annotations

import concurrent.futures
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtpgemm.so")
INCLUDE = os.path.join(ROOT, "include")
FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
         f"-I{INCLUDE}", f"-I{CSRC}"]

UNITS = [("tpgemm.o", "tpgemm.cu", []), ("stream_inst.o", "stream_inst.cu", []), ("mx_inst.o", "mx_inst.cu", []),
         ("fp4_nv.o", "fp4_inst.cu", ["-DTPG_FP4=1"]), ("fp4_mx.o", "fp4_inst.cu", ["-DTPG_FP4=2"])] + [
    (f"tiled_e{e}.o", "tiled_inst.cu", [f"-DTPG_EPI={e}"]) for e in range(6)] + [
    ("tiled_g0.o", "tiled_inst.cu", ["-DTPG_EPI=0", "-DTPG_GROUPED=1"])]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources():
    out = [os.path.join(INCLUDE, "tpgemm.h")]
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh")):
            out.append(os.path.join(CSRC, f))
    return out


def _compile(unit, verbose):
    obj, src, extra = unit
    cmd = [_nvcc(), *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", os.path.join(BUILD, obj)]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    return subprocess.run(cmd, capture_output=True, text=True), obj


def build(force: bool = False, verbose: bool = False) -> str:
    newest = max(os.path.getmtime(s) for s in sources())
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest:
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    workers = max(1, min(len(UNITS), os.cpu_count() or 1))
    with concurrent.futures.ThreadPoolExecutor(workers) as ex:
        results = list(ex.map(lambda u: _compile(u, verbose), UNITS))
    failed = [(r, o) for r, o in results if r.returncode != 0]
    for r, o in results:
        if verbose or r.returncode != 0:
            sys.stderr.write(f"--- {o}\n{r.stdout}{r.stderr}")
    if failed:
        raise RuntimeError("nvcc failed building " + ", ".join(o for _, o in failed))
    tmp = LIB + f".tmp{os.getpid()}"
    link = [_nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp,
            *[os.path.join(BUILD, o) for o, _, _ in UNITS]]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc failed linking libtpgemm.so")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
