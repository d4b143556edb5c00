"""include/kvc.h from plain C: a C program (tests/c_abi/roundtrip.c) includes the header, links libkvc.so and runs
create -> block claims -> slot mapping -> append -> decode, checked against a host computation in double precision.
Without a GPU the program is only compiled and linked (the header is valid C and every call it makes resolves)."""
import os
import shutil
import subprocess

import pytest

import paged_kv_cache_27_gb300 as kvc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "roundtrip.c")


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime_api.h")):
            return cand
    nv = shutil.which("nvcc")
    return os.path.dirname(os.path.dirname(os.path.realpath(nv))) if nv else None


def _build(tmp_path):
    cc = shutil.which("cc") or shutil.which("gcc")
    cuda = _cuda_home()
    if not cc or not cuda:
        pytest.skip("no C compiler or CUDA toolkit")
    libdir = os.path.dirname(kvc.lib_path())
    exe = str(tmp_path / "roundtrip")
    cmd = [cc, "-std=c99", "-O1", "-Wall", "-Werror", SRC, "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), "-L", libdir, "-lkvc", "-L", os.path.join(cuda, "lib64"), "-lcudart",
           "-lm", f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{os.path.join(cuda, 'lib64')}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_caller_compiles_and_links(tmp_path):
    assert os.path.exists(_build(tmp_path))


@pytest.mark.gpu
def test_c_caller_roundtrip(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c_abi_roundtrip ok" in r.stdout
