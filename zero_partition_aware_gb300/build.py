"""Builds libzr.so in-tree: the sm_103a kernels and the host C-ABI code.

Two translation units compiled in parallel by nvcc, linked with the static
CUDA runtime; a linker version script exports only the ``zr_*`` entry points
declared in ``include/zr.h``. The same kernels compiled with ZR_CHECKED (the
bounds-checked build, for tests) are linked into libzr_checked.so beside it.
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
LIB_CHECKED = os.path.join(OUT_DIR, "libzr_checked.so")
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
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [__file__]
    for lib in (LIB, LIB_CHECKED):
        if not os.path.exists(lib) or _foreign(lib):
            return True
        t = os.path.getmtime(lib)
        if any(os.path.getmtime(d) > t for d in deps):
            return True
    return False


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
        objs = {LIB: [], LIB_CHECKED: []}
        cmds = []
        for src in SOURCES:
            variants = [(LIB, []), (LIB_CHECKED, ["-DZR_CHECKED"])] if src.endswith(".cu") else [(None, [])]
            for lib, defs in variants:
                obj = os.path.join(tmp, src + ("_checked" if defs else "") + ".o")
                cmd = [nv, *COMMON, *defs, "-c", os.path.join(CSRC, src), "-o", obj]
                if src.endswith(".cu"):
                    cmd[1:1] = ARCH + ["-lineinfo"]
                    if ptxas_verbose and not defs:
                        cmd.insert(1, "-Xptxas=-v")
                for target in ([lib] if lib else [LIB, LIB_CHECKED]):
                    objs[target].append(obj)
                cmds.append(cmd)
        with ThreadPoolExecutor(len(cmds)) as ex:
            list(ex.map(lambda c: _run(c, verbose), cmds))
        vs = os.path.join(tmp, "exports.map")
        with open(vs, "w") as f:
            f.write("{ global: zr_*; local: *; };\n")
        for lib in (LIB, LIB_CHECKED):
            tmp_lib = lib + f".{os.getpid()}.tmp"
            _run([nv, *ARCH, "-shared", "-o", tmp_lib, *objs[lib], "-Xlinker", f"--version-script={vs}"], verbose)
            os.replace(tmp_lib, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))
