"""Build libdomino.so (the C-ABI CUDA library) in-tree for sm_103a.

Each translation unit under csrc/ is compiled in parallel with nvcc, then
linked into draft_head_gb300/lib/libdomino.so with the CUDA runtime linked
statically, so the library loads (and exports its symbols) on machines with
no GPU driver; the driver is only needed when a call runs.

    python -m draft_head_gb300.build [--force]
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "lib")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(OUT_DIR, "libdomino.so")
LIB_CHECKED = os.path.join(OUT_DIR, "libdomino_checked.so")  # -DDOMINO_CHECKED: device-side index checks
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    ds = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    ds.append(os.path.join(ROOT, "include", "domino.h"))
    return ds


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Build libdomino.so, or with checked=True libdomino_checked.so (the same
    sources compiled with -DDOMINO_CHECKED: device-side index checks that
    record DOMINO_ERR_INDEX and skip the access)."""
    out = LIB_CHECKED if checked else LIB
    if not force and up_to_date(out):
        return out
    bdir = os.path.join(BUILD_DIR, "checked") if checked else BUILD_DIR
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    flags = [ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
             "-Xptxas", "-v" if verbose else "-O3", "-I", os.path.join(ROOT, "include")]
    if checked:
        flags.append("-DDOMINO_CHECKED")

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, sources()))
    if verbose:
        for _, err in results:
            sys.stderr.write(err)
    objs = [o for o, _ in results]
    tmp = out + ".tmp"
    cmd = [nvcc, ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
