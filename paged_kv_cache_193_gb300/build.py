"""Build ``libpa.so`` (the C-ABI paged-attention library) for sm_103a.

Each ``csrc/*.cu`` file is compiled in parallel with nvcc, then linked into a
shared library with the CUDA runtime linked statically, so the library only
needs the driver at run time.  Output: ``paged_kv_cache_193_gb300/_build/libpa.so``.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libpa.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def _sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _sources() + _headers() + [__file__])


def compile_flags(verbose_ptxas: bool = False) -> list[str]:
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-I" + INCLUDE, "-I" + CSRC, "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]
    return flags


def build(force: bool = False, verbose_ptxas: bool = False, out: str | None = None,
          defines: tuple[str, ...] = ()) -> str:
    """Compile and link if any source is newer than the library; return its
    path.  ``out`` and ``defines`` (e.g. ``("PA_DECODE_WARPS=2",)``) build a
    variant of the library elsewhere, for launch-shape tuning."""
    lib = out or LIB
    if not force and not defines and out is None and not _stale():
        return LIB
    obj_dir = os.path.join(os.path.dirname(lib), os.path.basename(lib) + ".objs") if out else OUT_DIR
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()
    flags = compile_flags(verbose_ptxas) + ["-D" + d for d in defines]

    def one(src: str) -> tuple[str, str]:
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [cc, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(one, srcs))
    if verbose_ptxas:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
