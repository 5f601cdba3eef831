"""Build libmla.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

Every ``csrc/*.cu`` translation unit is compiled in parallel with nvcc for
``arch=compute_103a,code=sm_103a`` and linked into
``paged_mla_decode_gb300/libmla.so`` against the shared CUDA runtime (the same
``libcudart.so.13`` that PyTorch loads). Rebuilds only what changed.

Run ``python -m paged_mla_decode_gb300.build`` or call :func:`build`.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libmla.so")
# Test build: the FP8 decode kernel's QK issuer waits on a barrier that nothing
# completes and waits between roles give up after 20 ms, so that the timeout path
# (status bit, stop, drain, TMEM freed) can be run and checked. Not the product.
STALL_LIB_PATH = os.path.join(PKG, "libmla_stall_test.so")
STALL_DEFINES = ["-DMLA_TEST_STALL_QK", "-DMLA_PIPELINE_WAIT_NS=20000000ull"]

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libmla.so")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _deps(src: str):
    headers = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
    headers += glob.glob(os.path.join(INCLUDE, "*.h"))
    return [src] + headers


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(nvcc: str, src: str, verbose: bool, suffix: str = "", defines=()) -> str:
    obj = os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + suffix + ".o")
    if not _stale(obj, _deps(src)):
        return obj
    cmd = [nvcc, *ARCH_FLAGS, *NVCC_FLAGS, *defines, "-I", INCLUDE, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
    if verbose and res.stderr:
        sys.stderr.write(res.stderr)
    return obj


def _link(nvcc: str, path: str, objs) -> None:
    if not _stale(path, objs):
        return
    libdir = _cuda_lib_dir(nvcc)
    cmd = [nvcc, *ARCH_FLAGS, "-shared", "-cudart", "shared", "-o", path + ".tmp", *objs,
           "-Xlinker", f"-rpath,{libdir}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(path + ".tmp", path)


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile and link libmla.so (and the stall test library); return libmla.so's path."""
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    if force:
        for o in glob.glob(os.path.join(BUILD_DIR, "*.o")):
            os.remove(o)
    fp8 = os.path.join(CSRC, "decode_fp8.cu")
    jobs = [(src, "", ()) for src in srcs] + [(fp8, "_stall", tuple(STALL_DEFINES))]
    with cf.ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
        objs = list(ex.map(lambda j: _compile(nvcc, j[0], verbose, j[1], j[2]), jobs))
    product = objs[:len(srcs)]
    _link(nvcc, LIB_PATH, product)
    stall_obj = objs[len(srcs)]
    fp8_obj = os.path.join(BUILD_DIR, "decode_fp8.o")
    _link(nvcc, STALL_LIB_PATH, [o for o in product if o != fp8_obj] + [stall_obj])
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="--force" in sys.argv))
