"""Builds the CUDA library ``_build/libattn_gb300.so`` for sm_103a with nvcc.

Each translation unit compiles in parallel; the link uses the shared CUDA runtime
(so a process that already loaded it, e.g. through PyTorch, shares one runtime).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libattn_gb300.so")
SOURCES = ["attn_api.cu", "attn_fwd.cu", "attn_decode.cu", "attn_decode_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def cuda_home() -> str:
    env = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if env:
        return env
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "attn.h"), __file__]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link the library if any source is newer than it; returns its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = os.path.join(cuda_home(), "bin", "nvcc")
    if not os.path.exists(nvcc):
        nvcc = shutil.which("nvcc") or "nvcc"
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if verbose:
        common += ["-Xptxas", "-v"]
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(OUT_DIR, src.replace(".cu", f".{os.getpid()}.o"))
        objs.append(obj)
        cmd = [nvcc, *common, "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for cmd, pr in procs:
        out, _ = pr.communicate()
        if verbose and out:
            sys.stderr.write(out)
        if pr.returncode != 0:
            failed.append((cmd, out))
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + o for c, o in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    tmp = LIB + f".tmp{os.getpid()}"
    lib64 = os.path.join(cuda_home(), "lib64")
    subprocess.check_call([nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
                           "-Xlinker", "-rpath", "-Xlinker", lib64])
    os.replace(tmp, LIB)
    for o in objs:
        try:
            os.remove(o)
        except OSError:
            pass
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
