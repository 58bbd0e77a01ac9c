"""Build libtpmlp.so in-tree: nvcc for sm_103a only, one translation unit
per .cu file compiled in parallel, then a shared-library link.

build(debug=True) makes a second library, libtpmlp_debug.so (objects in
_build_debug), with the kernels' device-side index checks compiled in
(-DTP_DEVICE_CHECKS=1): a failed check is reported by tp_last_device_status
as TP_ERR_DEVICE_CHECK and the guarded access is skipped."""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libtpmlp.so")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libtpmlp_debug.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-I", INCLUDE, "-I", CSRC]
DEBUG_FLAGS = ["-DTP_DEVICE_CHECKS=1"]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    out = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    out += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return out


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, build_dir, flags, extra):
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    if _stale(obj, [src] + _headers()) or extra:
        cmd = [NVCC] + ARCH + FLAGS + list(flags) + list(extra) + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if r.stderr.strip():
            sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile every kernel file for sm_103a and link libtpmlp.so (or, with
    `debug`, libtpmlp_debug.so with the device-side checks)."""
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    flags = DEBUG_FLAGS if debug else []
    os.makedirs(build_dir, exist_ok=True)
    srcs = sources()
    if force:
        for f in os.listdir(build_dir):
            os.remove(os.path.join(build_dir, f))
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(lambda s: _compile(s, build_dir, flags, extra_flags), srcs))
    if _stale(lib, objs) or force or extra_flags:
        tmp = lib + f".{os.getpid()}.tmp"
        cmd = [NVCC] + ARCH + ["-shared", "-Xcompiler", "-fPIC", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, debug="--debug" in sys.argv))
