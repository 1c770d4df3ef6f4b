"""Build ``libmoe_pooled_wave.so`` in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` translation unit compiles to an object in parallel, then
one link makes the shared library next to this file.  No cmake; the only
tool is nvcc.  ``python -m moe_routing_capacity_gb300.build`` runs it.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoe_pooled_wave.so")
# the checked build: every kernel index verified before use (-DMOE_CHECK=1)
CHECK_LIB = os.path.join(HERE, "libmoe_pooled_wave_check.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(os.path.join(SRC, f) for f in os.listdir(SRC) if f.endswith(".cu"))


def _compile(src: str, out_dir: str = OUT, extra=()) -> tuple[str, str]:
    obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose: bool = False, lib_path: str = LIB, extra_flags=()) -> str:
    """Compile and link.  ``lib_path`` and ``extra_flags`` (e.g. -D tuning
    macros) let a variant be built somewhere else without touching the
    package's own library."""
    out_dir = OUT if lib_path == LIB else os.path.splitext(lib_path)[0] + "_obj"
    os.makedirs(out_dir, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(lambda f: _compile(f, out_dir, tuple(extra_flags)), srcs))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = lib_path + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


def build_checked(verbose: bool = False) -> str:
    """The library with the kernels' index checks compiled in."""
    return build(verbose, CHECK_LIB, ("-DMOE_CHECK=1",))


if __name__ == "__main__":
    if "--check" in sys.argv:
        print(build_checked(verbose="-v" in sys.argv))
    else:
        print(build(verbose="-v" in sys.argv))
