"""Build step for the CUDA library (libbsattn.so), in-tree, for sm_103a only.

The translation units are compiled in parallel with nvcc and linked into
_lib/libbsattn.so.  Nothing is installed; the library is loaded from here.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
_CSRC = os.path.join(_PKG, "csrc")
_INC = os.path.join(_ROOT, "include")
LIBDIR = os.path.join(_PKG, "_lib")
LIB = os.path.join(LIBDIR, "libbsattn.so")

SOURCES = ["api.cu", "plan.cu", "fwd_sm103.cu", "bwd_sm103.cu", "noalloc.cu", "pipeline.cu"]
HEADERS = ["ptx.cuh", "internal.h", "bwd.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(_CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(_INC, "bsattn.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), out: str | None = None) -> str:
    """Compile and link libbsattn.so if any source is newer than it.

    extra_flags: more nvcc flags (the tuner's -D settings of the kernels'
    build-time parameters); out: the library path (default LIB; the tuner
    builds each setting into its own file under LIBDIR/variants)."""
    lib = out or LIB
    if not force and not _stale(lib):
        return lib
    os.makedirs(os.path.dirname(lib), exist_ok=True)
    nvcc = _nvcc()
    objdir = os.path.join(os.path.dirname(lib), f"obj{os.getpid()}")
    os.makedirs(objdir, exist_ok=True)
    common = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-I", _INC, "-I", _CSRC, *extra_flags]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(objdir, os.path.splitext(src)[0] + ".o")
        cmd = common + ["-c", os.path.join(_CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    shutil.rmtree(objdir, ignore_errors=True)
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
