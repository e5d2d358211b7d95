"""Builds librlk.so (the sm_103a kernels and their C ABI) in-tree with nvcc.

Each translation unit compiles in parallel for sm_103a only; the objects are
linked into a shared library with the CUDA runtime linked statically, so the
library loads on a host without a GPU driver (its calls then report
RLK_ERR_UNSUPPORTED_DEVICE).

Two flavours of the same sources: librlk.so (release) and librlk_debug.so
(-DRLK_DEBUG: every kernel checks each global store against the extent of its
buffer and records violations in the device error word; the linear-logp kernels
record per-CTA phase timestamps).  Same ABI, same arithmetic.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "librlk.so")
FLAVORS = {"release": (LIB_PATH, []),
           "debug": (os.path.join(PKG_DIR, "librlk_debug.so"), ["-DRLK_DEBUG"])}

SOURCES = ["common.cu", "linear_logp.cu", "linear_logp_bwd.cu", "det_gemm.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("rlk_device.cuh", "rlk_pipeline.cuh", "rlk_solo.cuh", "rlk_internal.h")]
HEADERS.append(os.path.join(INCLUDE, "rlk.h"))

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-I" + INCLUDE, "-I" + CSRC,
]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librlk.so")
    return path


def _stale(lib_path: str) -> bool:
    if not os.path.exists(lib_path):
        return True
    t = os.path.getmtime(lib_path)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(flavor: str, verbose: bool):
    """Starts the nvcc processes of one flavour: [(source, process)], objects."""
    cc = nvcc()
    _, extra = FLAVORS[flavor]
    out_dir = os.path.join(BUILD_DIR, flavor)
    os.makedirs(out_dir, exist_ok=True)
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [cc, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                            text=True)))
    return procs, objs


def _link(flavor: str, objs):
    lib_path, _ = FLAVORS[flavor]
    tmp = lib_path + f".tmp{os.getpid()}"
    link = [nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-cudart", "static",
            *objs, "-o", tmp]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, lib_path)
    return lib_path


def build(force: bool = False, verbose: bool = False, flavors=("release", "debug")) -> str:
    """Compile and link every requested flavour whose sources changed (all translation
    units of all flavours in parallel); returns the release library's path."""
    todo = [f for f in flavors if force or _stale(FLAVORS[f][0])]
    started = [(f, *_compile(f, verbose)) for f in todo]
    errors = []
    for f, procs, objs in started:
        for src, p in procs:
            out, _ = p.communicate()
            if p.returncode != 0:
                errors.append(f"{f} {src}:\n{out}")
            elif verbose and out:
                print(out, file=sys.stderr)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    for f, _, objs in started:
        _link(f, objs)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
