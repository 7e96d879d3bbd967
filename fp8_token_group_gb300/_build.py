"""Build the CUDA library in-tree: nvcc for sm_103a only, one object per translation
unit (compiled in parallel), linked into ``libptgq.so`` next to this file."""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libptgq.so")
SOURCES = ["ptgq_api.cu", "ptgq_inst_bf16_flat.cu", "ptgq_inst_bf16_masked.cu",
           "ptgq_inst_fp16_flat.cu", "ptgq_inst_fp16_masked.cu", "ptgq_next.cu"]
HEADERS = ["ptgq_internal.h", "ptgq_kernel.cuh", "ptgq_device.cuh", "ptgq_math.cuh",
           "silu_tables.inc"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# No fast-math: IEEE division/reciprocal, no denormal flushing, and no implicit
# multiply-add contraction (the kernels write every fused multiply-add explicitly).
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-Xcompiler", "-fPIC",
                     "-cudart", "shared"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libptgq.so")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(os.path.dirname(HERE), "include", "ptgq.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    cc = nvcc()
    objdir = os.path.join(HERE, "_build")
    os.makedirs(objdir, exist_ok=True)

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [cc, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    # -Bsymbolic: the library's own references (kernel tables, template instances) bind to
    # its own definitions even when another library in the process defines the same names.
    r = subprocess.run([cc, *ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-Bsymbolic",
                        "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
