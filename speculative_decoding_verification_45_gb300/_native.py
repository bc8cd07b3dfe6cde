"""Build and load the sm_103a shared library (libspec_verify.so) in-tree."""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
CSRC = os.path.join(PKG, "csrc")
# The host unit plus one unit per (dtype, proposal form) of kernels: compiled in parallel.
SOURCES = [os.path.join(CSRC, f) for f in ("spec_verify.cu", "kernels_bf16.cu", "kernels_bf16_point.cu",
                                            "kernels_f32.cu", "kernels_f32_point.cu")]
HEADERS = [os.path.join(INCLUDE, "spec_verify.h"), os.path.join(CSRC, "spec_verify_kernels.cuh")]
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libspec_verify.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]

_lock = threading.Lock()
_lib = None


class Options(ctypes.Structure):
    """spec_verify_options of include/spec_verify.h."""

    _fields_ = [("cluster_size", ctypes.c_int), ("kernel", ctypes.c_int), ("counters", ctypes.c_void_p),
                ("accept_hist", ctypes.c_void_p)]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libspec_verify.so")


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in SOURCES + HEADERS)


def _run(cmd):
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    return res.stdout + res.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/*.cu for sm_103a (one nvcc per unit, in parallel) and link
    _build/libspec_verify.so."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if not force and not _stale():
        return LIB_PATH
    nvcc, tag = nvcc_path(), f"tmp{os.getpid()}"
    objs = [os.path.join(BUILD_DIR, os.path.basename(src)[:-3] + f".{tag}.o") for src in SOURCES]
    cmds = [[nvcc, "-O3", "-std=c++17", *ARCH_FLAGS, "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE,
             *(["-Xptxas=-v"] if verbose else []), "-c", "-o", obj, src] for src, obj in zip(SOURCES, objs)]
    tmp = LIB_PATH + f".{tag}"
    try:
        with ThreadPoolExecutor(max_workers=len(cmds)) as pool:
            logs = list(pool.map(_run, cmds))
        logs.append(_run([nvcc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs, "-ldl"]))
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    if verbose:
        print("".join(logs))
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def load() -> ctypes.CDLL:
    """Load the built library; raises if it has not been built (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: run __graft_entry__.build() (or "
                               "speculative_decoding_verification_45_gb300._native.build()) first")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i32 = ctypes.c_void_p, ctypes.c_int
        common = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp]
        lib.spec_verify.argtypes = common
        lib.spec_verify.restype = i32
        lib.spec_verify_debug.argtypes = common + [vp] * 7
        lib.spec_verify_debug.restype = i32
        lib.spec_verify_ex.argtypes = common + [vp]
        lib.spec_verify_ex.restype = i32
        lib.spec_ngram_propose.argtypes = [vp, ctypes.c_int64, vp, i32, i32, i32, i32, vp, vp, vp]
        lib.spec_ngram_propose.restype = i32
        lib.spec_sample.argtypes = [vp, vp, vp, vp, i32, i32, i32, vp, vp, vp]
        lib.spec_sample.restype = i32
        lib.spec_tree_verify.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp, vp, vp]
        lib.spec_tree_verify.restype = i32
        lib.spec_verify_launch_shape.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp]
        lib.spec_verify_launch_shape.restype = i32
        lib.spec_device_pointer.argtypes = [vp, ctypes.POINTER(ctypes.c_void_p)]
        lib.spec_device_pointer.restype = i32
        lib.spec_status_string.argtypes = [i32]
        lib.spec_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib
