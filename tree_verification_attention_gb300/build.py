"""Build ``libtva.so`` (the C-ABI library) in-tree with nvcc for sm_103a.

Every ``csrc/*.cu`` is compiled to an object in parallel, then linked into
``tree_verification_attention_gb300/libtva.so`` with the CUDA runtime linked statically
(so the library does not depend on which libcudart the host process loaded).  A stamp
of the sources and flags skips the build when nothing changed.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libtva.so")
# The checked build: the same sources with -DTVA_CHECKED (device-side index checks that
# record TVA_ERR_INVALID_ARG instead of touching memory out of bounds; see tva_common.cuh).
CHECKED_BUILD_DIR = os.path.join(PKG, "_build_checked")
CHECKED_LIB_PATH = os.path.join(PKG, "libtva_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
                 "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtva.so")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stamp() -> str:
    h = hashlib.sha256()
    h.update(" ".join(CFLAGS).encode())
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            p = os.path.join(d, f)
            if os.path.isfile(p):
                h.update(f.encode())
                with open(p, "rb") as fh:
                    h.update(fh.read())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags=None, checked: bool = False) -> str:
    """Compile and link; return the path of libtva.so (libtva_checked.so with checked=True)."""
    build_dir = CHECKED_BUILD_DIR if checked else BUILD_DIR
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    extra = list(extra_flags or []) + (["-DTVA_CHECKED"] if checked else [])
    os.makedirs(build_dir, exist_ok=True)
    stamp = _stamp() + ("|" + " ".join(extra) if extra else "")
    stamp_path = os.path.join(build_dir, "stamp")
    if not force and os.path.exists(lib_path) and os.path.exists(stamp_path):
        with open(stamp_path) as f:
            if f.read() == stamp:
                return lib_path
    nvcc = _nvcc()
    flags = CFLAGS + extra

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    srcs = _sources()
    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs + ["-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return lib_path


if __name__ == "__main__":
    print(build(verbose=True))
    print(build(verbose=True, checked=True))
