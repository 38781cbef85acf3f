"""Build libks.so (the C-ABI library and its sm_103a kernels) in-tree with nvcc.

Each translation unit compiles in parallel; the shared library links the CUDA runtime
dynamically (so a process that already loaded libcudart.so.13, as torch does, shares one
runtime with it) with an rpath to the toolkit for processes that did not.

    python -m row_wise_rmsnorm_ks_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libks.so")
SOURCES = ["ks_abi.cu", "ks_host.cu", "ks_noalloc.cu", "ks_ops.cu", "ks_launch_bf16.cu",
           "ks_launch_f16.cu", "ks_launch_f32.cu"]
HEADERS = ["ks_kernels.cuh", "ks_internal.h", "ks_ptx.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
              "-Xptxas", "-v", f"-I{os.path.join(ROOT, 'include')}"]


def _cuda_home() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home:
        return home
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _nvcc() -> str:
    return shutil.which("nvcc") or os.path.join(_cuda_home(), "bin", "nvcc")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps += [os.path.join(ROOT, "include", "ks.h"), os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(OUT_DIR, os.path.basename(src) + ".o")
    cmd = [_nvcc(), *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr  # ptxas -v reports go to stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libks.so if it is missing or older than its sources; return its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    objs = [o for o, _ in results]
    report = "\n".join(r for _, r in results)
    with open(os.path.join(OUT_DIR, "ptxas_report.txt"), "w") as f:
        f.write(report)
    if verbose:
        print(report)
    tmp = LIB + f".tmp{os.getpid()}"
    lib_dir = os.path.join(_cuda_home(), "lib64")
    cmd = [_nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           f"-L{lib_dir}", "-Xlinker", f"-rpath,{lib_dir}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
