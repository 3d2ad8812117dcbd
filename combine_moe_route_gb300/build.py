"""Build libmoeroute.so in-tree for sm_103a.

Each .cu translation unit under csrc/ is compiled by nvcc in parallel, then
linked into ``_build/libmoeroute.so`` (CUDA runtime linked statically, so the
library needs no libcudart at load time).  ``python -m
combine_moe_route_gb300.build`` runs it from the command line.
"""
from __future__ import annotations

import concurrent.futures as cf
import fcntl
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libmoeroute.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (CUDA toolkit required to build libmoeroute)")
    return cand


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hdrs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hdrs + sources() + [os.path.abspath(__file__)]


def library_path() -> str:
    return os.path.join(OUT_DIR, LIB_NAME)


def up_to_date() -> bool:
    lib = library_path()
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          out_dir: str | None = None, defines: tuple[str, ...] = ()) -> str:
    """Compile and link; return the library path.  Skips work when up to date.

    ``out_dir`` and ``defines`` (``NAME`` or ``NAME=VALUE``) build a separate
    copy of the library, e.g. one with the test-only hooks switched on; such a
    build is always redone."""
    if out_dir is None and not defines and not force and up_to_date():
        return library_path()
    default = out_dir is None and not defines
    out_dir = out_dir or OUT_DIR
    os.makedirs(out_dir, exist_ok=True)
    # one build of a folder at a time: parallel processes (test workers) would
    # otherwise write the same object files; a caller that waited finds the
    # library already up to date
    with open(os.path.join(out_dir, ".lock"), "w") as lock:
        try:
            fcntl.flock(lock, fcntl.LOCK_EX)
        except OSError:   # a file system without locks: build unlocked, as a single process would
            pass
        if default and not force and up_to_date():
            return library_path()
        return _compile_and_link(out_dir, ptxas_info, verbose, defines)


def _compile_and_link(out_dir: str, ptxas_info: bool, verbose: bool, defines: tuple[str, ...]) -> str:
    exe = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    extra += [f"-D{d}" for d in defines]

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [exe, *ARCH, *NVCC_FLAGS, *extra, "-I", INCLUDE, "-I", CSRC, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, sources()))
    if verbose or ptxas_info:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    target = os.path.join(out_dir, LIB_NAME)
    tmp = target + f".tmp{os.getpid()}"
    cmd = [exe, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, target)
    return target


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="-v" in sys.argv))
