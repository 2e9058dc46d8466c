"""Build libflce.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each .cu under csrc/ compiles to its own object in parallel; the objects link
into ``libflce.so`` next to this file with the CUDA runtime linked statically,
so the library loads on a machine without a GPU (the C-ABI symbol test) and
needs only the driver on a GPU machine.

``--debug`` builds ``libflce_debug.so`` instead: the same sources with FLCE_DEBUG=1,
which compiles in-kernel bounds checks of every TMA box and epilogue store (a
failing check is reported as FLCE_ERR_BOUNDS and the access skipped).

    python -m linear_cross_entropy_forward_gb300.build [--verbose-ptxas] [--force] [--debug]
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libflce.so")
DEBUG_BUILD_DIR = os.path.join(PKG_DIR, "_build_debug")
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "libflce_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found (set CUDA_HOME)")
    return found


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(ROOT, "include", "flce.h"))
    deps.append(os.path.abspath(__file__))
    return deps


def _up_to_date(lib_path: str) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose_ptxas: bool = False, quiet: bool = True,
          debug: bool = False) -> str:
    """Compile every CUDA source for sm_103a and link libflce.so (libflce_debug.so, with
    the in-kernel bounds checks, when debug is set); returns its path."""
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    if not force and not verbose_ptxas and _up_to_date(lib_path):
        return lib_path
    nvcc = nvcc_path()
    os.makedirs(build_dir, exist_ok=True)
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-I" + os.path.join(ROOT, "include"), "-I" + CSRC]
    if debug:
        flags += ["-DFLCE_DEBUG=1"]
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose_ptxas:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results]
    tmp = lib_path + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    if not quiet:
        print(f"built {lib_path}")
    return lib_path


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("--debug", action="store_true",
                    help="build libflce_debug.so (in-kernel bounds checks)")
    a = ap.parse_args()
    build(force=a.force, verbose_ptxas=a.verbose_ptxas, quiet=False, debug=a.debug)


if __name__ == "__main__":
    main()
