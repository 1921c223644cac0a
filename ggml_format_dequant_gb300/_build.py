"""Build libqmv.so in-tree for sm_103a: each translation unit compiled by nvcc
in parallel, then linked into one shared library (CUDA runtime linked
statically, so the library depends only on the driver).

Flavours: "" is the product library; "check" is the same sources compiled with
QMV_BOUNDS_CHECK, in which the matvec kernel tests every shared- and
global-memory access against its region and raises QMV_STATUS_OUT_OF_BOUNDS
instead of making one outside it (a separate file, for tests)."""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import platform
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
              "-Xptxas", "-v"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


FLAVOURS = {"": [], "check": ["-DQMV_BOUNDS_CHECK"],
            # the checking build with a planted fault (ring slots half as long as
            # planned), for the test that the checks fire
            "check_planted": ["-DQMV_BOUNDS_CHECK", "-DQMV_BOUNDS_CHECK_PLANT"]}


def lib_path(flavour: str = "") -> str:
    tag = f"_{flavour}" if flavour else ""
    return os.path.join(BUILD, f"libqmv{tag}_{platform.machine()}.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date(flavour: str = "") -> bool:
    out = lib_path(flavour)
    if not os.path.exists(out):
        return False
    t = os.path.getmtime(out)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, flavour: str = "") -> str:
    """Compile and link; returns the library path. Writes nvcc's -Xptxas -v
    report to _build/ptxas_<flavour>_<arch>.log (ptxas_<arch>.log for the
    product library)."""
    if flavour not in FLAVOURS:
        raise ValueError(f"unknown flavour {flavour!r}")
    out = lib_path(flavour)
    if not force and up_to_date(flavour):
        return out
    os.makedirs(BUILD, exist_ok=True)
    arch = platform.machine()
    tag = f"{flavour}_" if flavour else ""

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + f"_{tag}{arch}.o")
        cmd = [nvcc()] + ARCH + NVCC_FLAGS + FLAVOURS[flavour] + ["-I", INCLUDE, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, _sources()))
    with open(os.path.join(BUILD, f"ptxas_{tag}{arch}.log"), "w") as f:
        for obj, log in results:
            f.write(f"==== {os.path.basename(obj)}\n{log}\n")
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results] + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, out)
    if verbose:
        print(f"built {out}")
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))
