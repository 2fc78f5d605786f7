"""Builds libzr.so in-tree: the sm_103a kernels and the host C-ABI code.

Two translation units compiled in parallel by nvcc, linked with the static
CUDA runtime; a linker version script exports only the ``zr_*`` entry points
declared in ``include/zr.h``.
"""
from __future__ import annotations

import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libzr.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON_FLAGS = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC,-Wall"]
COMMON = COMMON_FLAGS + ["-I", INCLUDE, "-I", CSRC]

SOURCES = ["kernels.cu", "layout.cpp"]
HEADERS = [os.path.join(INCLUDE, "zr.h"), os.path.join(CSRC, "zr_internal.h"), os.path.join(CSRC, "zr_kernels.cuh")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _foreign(path: str) -> bool:
    """True if an ELF file was built for another machine (e.g. x86-64 vs aarch64)."""
    import platform
    want = {"x86_64": 62, "aarch64": 183, "arm64": 183}.get(platform.machine())
    try:
        with open(path, "rb") as f:
            head = f.read(20)
        return want is not None and int.from_bytes(head[18:20], "little") != want
    except OSError:
        return True


def _stale() -> bool:
    if not os.path.exists(LIB) or _foreign(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [__file__]
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"build step failed ({r.returncode}): {' '.join(cmd)}")
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile libzr.so if any source changed (or force). Returns its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    nv = nvcc()
    with tempfile.TemporaryDirectory(prefix="zr_build_") as tmp:
        objs, cmds = [], []
        for src in SOURCES:
            obj = os.path.join(tmp, src + ".o")
            cmd = [nv, *COMMON, "-c", os.path.join(CSRC, src), "-o", obj]
            if src.endswith(".cu"):
                cmd[1:1] = ARCH + ["-lineinfo"]
                if ptxas_verbose:
                    cmd.insert(1, "-Xptxas=-v")
            objs.append(obj)
            cmds.append(cmd)
        with ThreadPoolExecutor(len(cmds)) as ex:
            list(ex.map(lambda c: _run(c, verbose), cmds))
        vs = os.path.join(tmp, "exports.map")
        with open(vs, "w") as f:
            f.write("{ global: zr_*; local: *; };\n")
        tmp_lib = LIB + f".{os.getpid()}.tmp"
        _run([nv, *ARCH, "-shared", "-o", tmp_lib, *objs, "-Xlinker", f"--version-script={vs}"], verbose)
        os.replace(tmp_lib, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))
