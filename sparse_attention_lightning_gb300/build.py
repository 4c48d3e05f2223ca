"""Build libdsa.so in-tree for sm_103a (GB300).

    python -m sparse_attention_lightning_gb300.build [--verbose] [--checked]

Each .cu under csrc/ compiles to an object in parallel (nvcc, one -gencode for
compute_103a/sm_103a), then the objects link into
sparse_attention_lightning_gb300/libdsa.so against the CUDA runtime.  ptxas
resource usage (-Xptxas -v) is written to _build/ptxas.log.  --checked builds
libdsa_checked.so instead (-DDSA_CHECKED: the kernels test their internal
invariants on the device and report failures through the status word), in
_build_checked/.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdsa.so")
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libdsa_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return ["-O3", "-std=c++17", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC,-O2",
            "-I", os.path.join(ROOT, "include"), "-I", CSRC, "--expt-relaxed-constexpr",
            "-Xptxas", "-v", *extra]


def _compile(src: str, extra, bdir: str) -> tuple:
    obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *_flags(extra), "-c", src, "-o", obj]
    p = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, p.returncode, p.stdout + p.stderr


def build(verbose: bool = False, extra=(), checked: bool = False) -> str:
    bdir, lib = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    if checked:
        extra = (*extra, "-DDSA_CHECKED")
    os.makedirs(bdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = srcs + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    if os.path.exists(lib) and (checked or not extra):
        lib_m = os.path.getmtime(lib)
        if all(os.path.getmtime(d) < lib_m for d in deps):
            return lib
    logs = []
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda s: _compile(s, extra, bdir), srcs))
    failed = [r for r in results if r[2] != 0]
    for src, _, rc, log in results:
        logs.append(f"== {os.path.basename(src)} (rc={rc})\n{log}")
    with open(os.path.join(bdir, "ptxas.log"), "w") as f:
        f.write("\n".join(logs))
    if failed:
        msg = "\n".join(f"{os.path.basename(s)}:\n{log}" for s, _, _, log in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    tmp = lib + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[r[1] for r in results], "-lcudart"]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError("link failed:\n" + p.stdout + p.stderr)
    os.replace(tmp, lib)
    if verbose:
        print("\n".join(logs))
    return lib


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--checked", action="store_true")
    a = ap.parse_args()
    print(build(verbose=a.verbose, checked=a.checked))
    sys.exit(0)
