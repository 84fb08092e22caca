"""Builds the CUDA library ``libfa_gb300.so`` (in-tree, beside this file).

Every ``csrc/*.cu`` translation unit is compiled for sm_103a only, in parallel,
then linked into one shared library with the CUDA runtime linked statically,
so the C ABI of ``include/fa.h`` is the only interface.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libfa_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
                   f"-I{CSRC}", f"-I{os.path.join(os.path.dirname(HERE), 'include')}"] + list(extra)


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib_path: str = LIB_PATH) -> str:
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = srcs + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + [
        os.path.join(os.path.dirname(HERE), "include", "fa.h")]
    newest = max(os.path.getmtime(p) for p in deps)
    if not force and not extra_flags and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= newest:
        return lib_path
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = nvcc_path()
    tag = "x".join(f for f in extra_flags).replace("-", "").replace("=", "") or "default"
    if len(tag) > 64:  # keep object names within the file system's limit
        tag = "v" + hashlib.sha256(tag.encode()).hexdigest()[:16]

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + f".{tag}.o")
        cmd = [nvcc] + _flags(extra_flags) + ["-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib_path + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs,
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys

    print(build(force=True, verbose="-v" in sys.argv))
