"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle harness.

Holds no arithmetic of the method itself: only the counter-based generator
(splitmix64 + Box-Muller, see ``synth.c``) and the recipes that turn it into
the workloads' lengths, block tables and bf16 values.  Both the CUDA path and
the oracle consume what this module produces; neither imports the other.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None


def build_command(out_path: str = _LIB_PATH) -> list[str]:
    return ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
            os.path.join(_HERE, "synth.c"), "-o", out_path, "-lm"]


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(os.path.join(_HERE, "synth.c")):
        os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(build_command(tmp))
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        u64, i64, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        L.synth_key.restype = u64
        L.synth_key.argtypes = [u64, u64]
        L.synth_u64.restype = u64
        L.synth_u64.argtypes = [u64, u64]
        L.synth_normal.restype = ctypes.c_double
        L.synth_normal.argtypes = [u64, u64]
        L.synth_bf16_from_double.restype = ctypes.c_uint16
        L.synth_bf16_from_double.argtypes = [ctypes.c_double]
        for name in ("synth_fill_normal_bf16", "synth_fill_normal_f64",
                     "synth_fill_uniform_f64", "synth_fill_u64"):
            f = getattr(L, name)
            f.restype = None
            f.argtypes = [u64, u64, u64, i64, vp]
        L.synth_permutation.restype = None
        L.synth_permutation.argtypes = [u64, u64, i64, vp]
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ---------------------------------------------------------------- primitives
def normal_bf16(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    """n draws of N(0,1) rounded to bf16, as uint16 bit patterns."""
    out = np.empty(int(n), dtype=np.uint16)
    if n:
        lib().synth_fill_normal_bf16(seed, stream, offset, int(n), _ptr(out))
    return out


def normal_f64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(int(n), dtype=np.float64)
    if n:
        lib().synth_fill_normal_f64(seed, stream, offset, int(n), _ptr(out))
    return out


def uniform_f64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(int(n), dtype=np.float64)
    if n:
        lib().synth_fill_uniform_f64(seed, stream, offset, int(n), _ptr(out))
    return out


def u64(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(int(n), dtype=np.uint64)
    if n:
        lib().synth_fill_u64(seed, stream, offset, int(n), _ptr(out))
    return out


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(int(n), dtype=np.int32)
    if n:
        lib().synth_permutation(seed, stream, int(n), _ptr(out))
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact; a harness convenience)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def stream_id(*parts: int) -> int:
    """Pack small non-negative integers into one 64-bit stream id."""
    s = 0
    for p in parts:
        s = (s * 1_000_003 + int(p) + 1) & 0xFFFFFFFFFFFFFFFF
    return s


from .workloads import Workload, make_workload, WORKLOADS  # noqa: E402,F401
