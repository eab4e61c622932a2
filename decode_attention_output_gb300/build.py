"""Builds libdecode_attn.so in-tree for sm_103a with nvcc (no cmake, no torch).

Each .cu file compiles in its own nvcc process (in parallel), then one link
step produces ``_lib/libdecode_attn.so``. A stamp of the sources, headers and
flags skips the build when nothing changed.

``build(checked=True)`` makes the bounds-checked copy instead,
``_lib/checked/libdecode_attn_checked.so`` (compiled with -DDA_BOUNDS_CHECK: every
guarded index is tested against its buffer and a failure is recorded in the device
error word); the tests load it beside the regular library.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_NAME = "libdecode_attn.so"
CHECKED_NAME = "libdecode_attn_checked.so"
CHECKED_FLAGS = ["-DDA_BOUNDS_CHECK"]
SOURCES = ["api.cu", "attn_decode.cu", "attn_decode_d256.cu", "attn_decode_paged.cu", "attn_decode_fp8.cu",
           "oproj_gemv.cu", "oproj_umma.cu", "oproj_onchip.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def lib_path(checked: bool = False) -> str:
    if checked:
        return os.path.join(LIB_DIR, "checked", CHECKED_NAME)
    return os.path.join(LIB_DIR, LIB_NAME)


def _stamp(extra=()) -> str:
    h = hashlib.sha1()
    for d in (CSRC, INCLUDE):
        for name in sorted(os.listdir(d)):
            if name.endswith((".cu", ".cuh", ".h")):
                with open(os.path.join(d, name), "rb") as f:
                    h.update(name.encode() + f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS + list(extra)).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = False) -> str:
    """Compile and link the library (or its bounds-checked copy); returns its path."""
    if checked:
        extra_flags = [*CHECKED_FLAGS, *extra_flags]
    out = lib_path(checked)
    out_dir = os.path.dirname(out)
    obj_dir = os.path.join(out_dir, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    stamp = _stamp(extra_flags)
    stamp_file = os.path.join(out_dir, "stamp.txt")
    if not force and os.path.exists(out) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return out
    exe = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        cmd = [exe, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr, file=sys.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = out + f".tmp{os.getpid()}"
    cmd = [exe, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, out)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))
