"""Build libattn_fwd.so (forward and backward kernels) in-tree with nvcc for sm_103a (GB300)."""
from __future__ import annotations

import fcntl
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SOURCES = [os.path.join(PKG, "csrc", "attn_fwd.cu"), os.path.join(PKG, "csrc", "attn_fwd_wide.cu"),
           os.path.join(PKG, "csrc", "attn_bwd.cu")]
HEADERS = [os.path.join(ROOT, "include", "attn_fwd.h"), os.path.join(ROOT, "include", "attn_bwd.h"),
           os.path.join(PKG, "csrc", "attn_wide.h"), os.path.join(PKG, "csrc", "tc_sm103.cuh")]
LIB_PATH = os.path.join(PKG, "libattn_fwd.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC",
]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise FileNotFoundError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def _stale(out: str) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(f) > t for f in SOURCES + HEADERS)


def build_library(force: bool = False, extra_flags=(), out: str = LIB_PATH) -> str:
    """Compile the CUDA sources into ``out`` unless it is newer than every source."""
    lock_path = out + ".lock"
    with open(lock_path, "w") as lk:
        fcntl.flock(lk, fcntl.LOCK_EX)
        if not force and not _stale(out):
            return out
        tmp = out + f".tmp{os.getpid()}"
        nvcc = nvcc_path()
        # one nvcc per translation unit, all at once, then one link
        objs = [f"{tmp}.{os.path.splitext(os.path.basename(src))[0]}.o" for src in SOURCES]
        procs = []
        for src, obj in zip(SOURCES, objs):
            cmd = [nvcc, *NVCC_FLAGS, *extra_flags, "-I", os.path.join(ROOT, "include"), "-c", "-o", obj, src]
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)))
        try:
            for cmd, proc in procs:
                stdout, stderr = proc.communicate()
                if proc.returncode != 0:
                    raise RuntimeError(f"nvcc failed ({proc.returncode}):\n{' '.join(cmd)}\n{stdout}\n{stderr}")
            cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp, *objs]
            res = subprocess.run(cmd, capture_output=True, text=True)
            if res.returncode != 0:
                raise RuntimeError(f"nvcc link failed ({res.returncode}):\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
            os.replace(tmp, out)
        finally:
            for _, proc in procs:
                if proc.poll() is None:
                    proc.kill()
                    proc.wait()
            for obj in objs:
                if os.path.exists(obj):
                    os.remove(obj)
    return out
