"""Build the CUDA library libkvc.so in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel; the shared object links the CUDA
runtime dynamically so that it shares the runtime instance already loaded by
PyTorch.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "lib")
LIB = os.path.join(OUT_DIR, "libkvc.so")
SOURCES = ["api.cu", "append.cu", "decode.cu", "group.cu", "group_tc.cu", "multi_tc.cu", "prefill.cu",
           "prefill_1t.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-Wall", "-cudart", "shared"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _cuda_lib_dir(nv: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nv))), "lib64")


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile libkvc.so; KVC_NVCC_FLAGS (environment) adds nvcc flags, e.g. -D tuning knobs."""
    extra_flags = list(extra_flags) + os.environ.get("KVC_NVCC_FLAGS", "").split()
    os.makedirs(OUT_DIR, exist_ok=True)
    stamp = LIB + ".flags"
    flags_id = " ".join(extra_flags)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(os.path.dirname(HERE), "include", "kvc.h"))
    if not force and os.path.exists(LIB) and os.path.exists(stamp):
        newest = max(os.path.getmtime(d) for d in deps)
        with open(stamp) as f:
            same_flags = f.read() == flags_id
        if same_flags and os.path.getmtime(LIB) >= newest:
            return LIB
    nv = nvcc()
    objdir = os.path.join(OUT_DIR, "obj")
    os.makedirs(objdir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(objdir, src.replace(".cu", ".o"))
        cmd = [nv, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nv, *ARCH, "-shared", "-cudart", "shared", *objs, "-o", tmp,
           "-Xlinker", f"-rpath,{_cuda_lib_dir(nv)}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(flags_id)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
