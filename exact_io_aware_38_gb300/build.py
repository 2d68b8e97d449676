"""Builds libfa.so in-tree from csrc/*.cu for sm_103a (nvcc only, translation units in parallel).

Usage: python -m exact_io_aware_38_gb300.build [--debug-bounds]
"""

from __future__ import annotations

import glob
import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"),
                   "--expt-relaxed-constexpr"] + list(extra)


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _digest(extra) -> str:
    h = hashlib.sha256()
    for p in _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + [os.path.join(ROOT, "include", "fa.h")]:
        h.update(p.encode())
        h.update(open(p, "rb").read())
    h.update(" ".join(_flags(extra)).encode())
    h.update(nvcc().encode())
    return h.hexdigest()


def build(extra=(), verbose=False, force=False) -> str:
    """Compile every csrc/*.cu and link libfa.so; skips the work if sources and flags are unchanged."""
    os.makedirs(OUT_DIR, exist_ok=True)
    stamp = os.path.join(OUT_DIR, "stamp")
    dig = _digest(extra)
    if not force and os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == dig:
        return LIB
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(OUT_DIR, os.path.basename(src)[:-3] + ".o")
        cmd = [cc] + _flags(extra) + ["-c", src, "-o", obj]
        if verbose:
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    srcs = _sources()
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB + ".tmp"
    r = subprocess.run([cc] + ARCH + ["-shared", "-o", tmp] + objs, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(dig)
    return LIB


TEST_WITHHOLD_LIB = os.path.join(OUT_DIR, "libfa_withhold_kv.so")


def build_withhold_kv_test_lib() -> str:
    """Test-only variant whose forward producer never loads K/V and whose waits give up after
    50 ms: used to check that a wait that runs out returns FA_ERR_DEVICE_TIMEOUT cleanly."""
    os.makedirs(OUT_DIR, exist_ok=True)
    cc = nvcc()
    extra = ["-DFA_TEST_WITHHOLD_KV"]
    objs = []
    for src in _sources():
        obj = os.path.join(OUT_DIR, "withhold_" + os.path.basename(src)[:-3] + ".o")
        r = subprocess.run([cc] + _flags(extra) + ["-c", src, "-o", obj], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        objs.append(obj)
    r = subprocess.run([cc] + ARCH + ["-shared", "-o", TEST_WITHHOLD_LIB] + objs, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return TEST_WITHHOLD_LIB


if __name__ == "__main__":
    extra = ["-DFA_DEBUG_BOUNDS"] if "--debug-bounds" in sys.argv else []
    print(build(extra, verbose="-v" in sys.argv, force=True))
