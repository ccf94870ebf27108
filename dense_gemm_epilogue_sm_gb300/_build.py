"""Builds ``libgemm_sm103.so`` in-tree with nvcc for sm_103a only.

Three translation units compile in parallel into ``_build/`` and link into
one shared library next to this file.  The CUDA runtime is linked
statically (nvcc's default), so the library needs only the NVIDIA driver at
run time; the driver's tensor-map encoder is looked up through the runtime.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libgemm_sm103.so")
# Diagnostic builds, each a library of its own (select one at run time with
# GEMM_SM103_LIBRARY): "debug" checks every store index in the kernel
# (GEMM_DEBUG), "stamps" records %globaltimer at fixed points (GEMM_STAMPS).
VARIANTS = {"": [], "debug": ["-DGEMM_DEBUG"], "stamps": ["-DGEMM_STAMPS"]}


def library_path(variant=""):
    return LIB if not variant else os.path.join(HERE, f"libgemm_sm103_{variant}.so")
SOURCES = ["gemm_ob2.cu", "gemm_ob4.cu", "gemm_ob1.cu", "gemm_sm103.cu", "api.cpp", "layout_api.cu", "noalloc.cu",
           "reduce_finish.cu"]
HEADERS = ["gemm_internal.h", "gemm_kernel.cuh", "gemm_variants.h", "layout.hpp", "ptx.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the GEMM library")


def _inputs():
    inc = os.path.join(os.path.dirname(HERE), "include")
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files += [os.path.join(inc, f) for f in os.listdir(inc)]
    files.append(os.path.abspath(__file__))
    return files


def _stale(lib):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, variant: str = "") -> str:
    lib = library_path(variant)
    if not force and not _stale(lib):
        return lib
    nvcc = _nvcc()
    build_dir = BUILD if not variant else f"{BUILD}_{variant}"
    os.makedirs(build_dir, exist_ok=True)
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                     "-I", os.path.join(os.path.dirname(HERE), "include")] + VARIANTS[variant]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            print(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    variant = next((a.split("=", 1)[1] for a in sys.argv[1:] if a.startswith("--variant=")), "")
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, variant=variant))
