"""Compile tests/c_abi/roundtrip.c (plain C, the public header and the CUDA runtime API only)
against the built library."""
import glob
import os
import shutil
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "roundtrip.c")


def cuda_root() -> str:
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def cudart_dir(root: str) -> str:
    for d in [os.path.join(root, "lib64"), os.path.join(root, "lib")] + glob.glob(os.path.join(root, "targets", "*", "lib")):
        if glob.glob(os.path.join(d, "libcudart.so*")):
            return d
    raise FileNotFoundError("libcudart.so not found under " + root)


def compile_roundtrip(lib_path: str, out_dir: str) -> str:
    root = cuda_root()
    exe = os.path.join(out_dir, "c_abi_roundtrip")
    lib_dir = os.path.dirname(lib_path)
    rt_dir = cudart_dir(root)
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", SRC,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(root, "include"),
           "-L", lib_dir, "-l:" + os.path.basename(lib_path), "-L", rt_dir, "-lcudart", "-lm",
           "-Wl,-rpath," + lib_dir, "-Wl,-rpath," + rt_dir, "-o", exe]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return exe
