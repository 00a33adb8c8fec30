"""Build libkvb.so in-tree for sm_103a with nvcc (no cmake, no torch extension machinery).

    python -m kv_buffered_decoding_gb300.build [--force]

Each translation unit compiles in its own nvcc/g++ process, in parallel; the
objects are linked into ``kv_buffered_decoding_gb300/_lib/libkvb.so`` with the
CUDA runtime linked statically, so the library depends only on the driver.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libkvb.so")

CU_SOURCES = ["decode.cu", "decode_stream.cu", "short.cu", "verify.cu", "verify_tc.cu", "flush.cu",
              "baseline.cu", "prefill.cu", "prefill_tc.cu"]
CPP_SOURCES = ["kvb_host.cpp", "device_setup.cpp"]
HEADERS = ["kvb_internal.h", "kvb_device.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> str:
    env = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if env:
        return env
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _nvcc() -> str:
    return os.path.join(cuda_home(), "bin", "nvcc")


def _inputs():
    files = [os.path.join(CSRC, f) for f in CU_SOURCES + CPP_SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "kvb.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _run(cmd):
    proc = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    return cmd, proc.returncode, proc.stdout


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False,
          defines=(), out_dir: str | None = None) -> str:
    """Compile every kernel for sm_103a and link libkvb.so; return its path.

    ``defines`` (e.g. ``["KVB_DECODE_SPLIT=1"]``) and ``out_dir`` build a variant of
    the library elsewhere without touching the in-tree one.
    """
    lib = LIB if out_dir is None else os.path.join(out_dir, "libkvb.so")
    out_dir = OUT_DIR if out_dir is None else out_dir
    if not force and not defines and lib == LIB and up_to_date():
        return LIB
    os.makedirs(out_dir, exist_ok=True)
    obj_dir = os.path.join(out_dir, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    inc = ["-I", INCLUDE, "-I", CSRC] + [f"-D{d}" for d in defines]
    jobs = []
    objs = []
    for src in CU_SOURCES:
        obj = os.path.join(obj_dir, src + ".o")
        objs.append(obj)
        cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
               "--expt-relaxed-constexpr", *inc, "-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_verbose:
            cmd.insert(1, "-Xptxas=-v")
        jobs.append(cmd)
    for src in CPP_SOURCES:
        obj = os.path.join(obj_dir, src + ".o")
        objs.append(obj)
        cxx = os.environ.get("CXX", "g++")
        jobs.append([cxx, "-O2", "-std=c++17", "-fPIC", "-Wall", *inc,
                     "-I", os.path.join(cuda_home(), "include"), "-c",
                     os.path.join(CSRC, src), "-o", obj])
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(_run, jobs))
    failed = [(c, out) for c, rc, out in results if rc != 0]
    if verbose or ptxas_verbose:
        for c, rc, out in results:
            print(" ".join(c))
            print(out)
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + out for c, out in failed)
        raise RuntimeError(f"libkvb build failed:\n{msg}")
    tmp = lib + ".tmp"
    link = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    cmd, rc, out = _run(link)
    if rc != 0:
        raise RuntimeError("libkvb link failed:\n" + " ".join(cmd) + "\n" + out)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    path = build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                 ptxas_verbose="--ptxas" in sys.argv)
    print(path)
