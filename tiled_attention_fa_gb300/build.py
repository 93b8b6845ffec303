"""Build the C-ABI shared library in-tree with nvcc (sm_103a only).

    python -m tiled_attention_fa_gb300.build          # builds libfa_gb300.so next to this file

Each .cu unit compiles in parallel to an object file under ``_build/``; the
objects then link into ``libfa_gb300.so`` with the CUDA runtime linked
statically, so loading the library needs no GPU and no libcuda at load time.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB_NAME = "libfa_gb300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
UNITS = ["api.cu", "fwd.cu", "bwd.cu", "decode.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")


def _flags(verbose_ptxas: bool) -> list:
    f = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _compile(unit: str, verbose_ptxas: bool) -> tuple:
    src = os.path.join(CSRC, unit)
    obj = os.path.join(BUILD, unit.replace(".cu", ".o"))
    cmd = [nvcc(), "-c", src, "-o", obj] + _flags(verbose_ptxas)
    r = subprocess.run(cmd, capture_output=True, text=True)
    return unit, obj, r.returncode, r.stdout + r.stderr


def build(verbose_ptxas: bool = False, quiet: bool = False) -> str:
    """Compile every unit and link the shared library; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        results = list(ex.map(lambda u: _compile(u, verbose_ptxas), UNITS))
    failed = [r for r in results if r[2] != 0]
    for unit, _, rc, out in results:
        if (rc != 0 or verbose_ptxas) and out.strip():
            print(f"---- {unit} (rc={rc})\n{out}", file=sys.stderr)
    if failed:
        raise RuntimeError("nvcc failed for " + ", ".join(r[0] for r in failed))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc(), "-shared", "-o", tmp] + [r[1] for r in results] + ARCH + \
        ["-Xcompiler", "-fPIC", "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB_PATH)
    if not quiet:
        print("built", LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(verbose_ptxas="-v" in sys.argv)
