"""CPU oracle for the paged KV-cache decode step -- TEST INFRASTRUCTURE ONLY.

A plain fp64 C implementation (``kvc_oracle.c``) of what the hot path
computes, reached through ctypes with numpy arrays.  Only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg (and its
``--impl reference`` arm) may import this package; the CUDA library never
does, and the two share no code.

Functions and the passages they follow (page titles; the C file has details):
  kv_bytes, kv_bytes_growth   "KV cache: Generation state, latency, and
                              allocation" Eq. 21.2, Eq. 21.3
  locate                      same page, 21.5 and Table 21.1
  write_tokens / append       same page, Eq. 21.6 and Table 21.1 steps 1-2
  gather                      same page, 21.5 (attention follows the table)
  e4m3_encode / e4m3_decode   OCP FP8 E4M3 definition; "KV Cache Explained",
                              "What changes when you use FP8 KV"
  fp8_scales                  absmax over positions / 448 (the fp8 workload's
                              stated calibration)
  decode, prefill             same page 21.1 (score normalisation and value
                              mixture over every cached key plus the new one;
                              GQA/MQA head sharing), 21.3 chunked prefill
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import time

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvc_oracle.c")
LIB_PATH = os.path.join(_HERE, "_build", "libkvc_oracle.so")

OK, ERR_ARG, ERR_BAD_BLOCK, ERR_RANGE = 0, 1, 3, 4
KIND_E4M3, KIND_BF16, KIND_INT4 = 1, 2, 3       # stored-scalar kinds (same codes as the C file)

_lib = None


def build_command(out_path: str = LIB_PATH, mutant: int = 0) -> list[str]:
    extra = [f"-DORC_MUTANT={mutant}"] if mutant else []
    return ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", *extra, _SRC, "-o", out_path, "-lm"]


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(LIB_PATH), exist_ok=True)
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(build_command(tmp))
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def lib():
    global _lib
    if _lib is None:
        # KVC_ORACLE_LIB: a build of this source with a planted mistake (the mutation test)
        path = os.environ.get("KVC_ORACLE_LIB") or build()
        L = ctypes.CDLL(path)
        i64, i32, u64, vp, dbl = ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64, ctypes.c_void_p, ctypes.c_double
        L.orc_kv_bytes.restype = u64
        L.orc_kv_bytes.argtypes = [i64] * 6
        L.orc_kv_bytes_growth.restype = u64
        L.orc_kv_bytes_growth.argtypes = [i64] * 5
        L.orc_bf16_to_double.restype = dbl
        L.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        L.orc_e4m3_to_double.restype = dbl
        L.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
        L.orc_e4m3_from_float.restype = ctypes.c_uint8
        L.orc_e4m3_from_float.argtypes = [ctypes.c_float]
        L.orc_fp8_scales.restype = None
        L.orc_fp8_scales.argtypes = [vp, i64, i32, i32, vp]
        L.orc_quantize_e4m3.restype = None
        L.orc_quantize_e4m3.argtypes = [vp, i64, i32, i32, vp, vp]
        L.orc_quantize_int4.restype = None
        L.orc_quantize_int4.argtypes = [vp, i64, i32, i32, vp, vp]
        L.orc_int4_encode.restype = ctypes.c_uint8
        L.orc_int4_encode.argtypes = [ctypes.c_float]
        L.orc_int4_decode.restype = dbl
        L.orc_int4_decode.argtypes = [ctypes.c_uint8]
        L.orc_int4_scales.restype = None
        L.orc_int4_scales.argtypes = [vp, i64, i32, i32, vp]
        L.orc_locate.restype = ctypes.c_int
        L.orc_locate.argtypes = [vp, i32, i64, i32, i64, vp, vp]
        L.orc_pool_offset.restype = u64
        L.orc_pool_offset.argtypes = [i64, i32, i32, i32, i32, i64, i32, i32, i32, i32]
        L.orc_write_tokens.restype = ctypes.c_int
        L.orc_write_tokens.argtypes = [vp, i64, i32, i32, i32, i32, i32, vp, i32, i32, vp, vp, vp, vp, vp]
        L.orc_gather.restype = ctypes.c_int
        L.orc_gather.argtypes = [vp, i64, i32, i32, i32, i32, i32, vp, i32, i64, vp, vp]
        L.orc_decode.restype = ctypes.c_int
        L.orc_decode.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, dbl, vp, vp]
        L.orc_prefill.restype = ctypes.c_int
        L.orc_prefill.argtypes = [vp, i64, vp, vp, i64, i32, i32, i32, i32, vp, dbl, vp, vp]
        L.orc_num_threads.restype = ctypes.c_int
        L.orc_num_threads.argtypes = []
        _lib = L
    return _lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous numpy"
    return a.ctypes.data


def num_threads() -> int:
    return int(lib().orc_num_threads())


# ------------------------------------------------------------------ bytes
def kv_bytes(L, B, H_KV, T, d_h, s) -> int:
    return int(lib().orc_kv_bytes(L, B, H_KV, T, d_h, s))


def kv_bytes_growth(L, B, H_KV, d_h, s) -> int:
    return int(lib().orc_kv_bytes_growth(L, B, H_KV, d_h, s))


# ------------------------------------------------------------------ scalars
def bf16_to_double(bits: int) -> float:
    return float(lib().orc_bf16_to_double(int(bits)))


def e4m3_decode(code: int) -> float:
    return float(lib().orc_e4m3_to_double(int(code)))


def e4m3_encode(x: float) -> int:
    return int(lib().orc_e4m3_from_float(float(x)))


def fp8_scales(x_bits: np.ndarray) -> np.ndarray:
    """x_bits: bf16 [n_tokens][H_KV][d_h] -> fp32 [H_KV][d_h] = absmax / 448."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    n, H, d = x_bits.shape
    out = np.empty((H, d), dtype=np.float32)
    lib().orc_fp8_scales(_p(x_bits), n, H, d, _p(out))
    return out


def quantize_e4m3(x_bits: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """bf16 [n][H_KV][d_h] -> e4m3 codes under fp32 scales [H_KV][d_h] (the append's rule)."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    n, H, d = x_bits.shape
    sc = np.ascontiguousarray(scales, dtype=np.float32).reshape(H, d)
    out = np.empty((n, H, d), dtype=np.uint8)
    lib().orc_quantize_e4m3(_p(x_bits), n, H, d, _p(sc), _p(out))
    return out


def int4_encode(y: float) -> int:
    return int(lib().orc_int4_encode(float(y)))


def int4_decode(nibble: int) -> float:
    return float(lib().orc_int4_decode(int(nibble)))


def int4_scales(x_bits: np.ndarray) -> np.ndarray:
    """x_bits: bf16 [n_tokens][H_KV][d_h] -> fp32 [H_KV][d_h] = absmax / 7."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    n, H, d = x_bits.shape
    out = np.empty((H, d), dtype=np.float32)
    lib().orc_int4_scales(_p(x_bits), n, H, d, _p(out))
    return out


def quantize_int4(x_bits: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """bf16 [n][H_KV][d_h] -> int4 nibbles (one per byte) under fp32 scales [H_KV][d_h]."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    n, H, d = x_bits.shape
    sc = np.ascontiguousarray(scales, dtype=np.float32).reshape(H, d)
    out = np.empty((n, H, d), dtype=np.uint8)
    lib().orc_quantize_int4(_p(x_bits), n, H, d, _p(sc), _p(out))
    return out


def kind_of(elem) -> int:
    """2 / 'bf16' -> bf16, 1 / 'fp8' -> e4m3, 'int4' -> int4."""
    return {2: KIND_BF16, "bf16": KIND_BF16, 1: KIND_E4M3, "fp8": KIND_E4M3, "e4m3": KIND_E4M3,
            "int4": KIND_INT4, KIND_INT4: KIND_INT4}[elem]


# ------------------------------------------------------------------ tables
def locate(bt_row: np.ndarray, t: int, bs: int, num_blocks: int):
    """(status, physical block, slot) of logical position t."""
    bt_row = np.ascontiguousarray(bt_row, dtype=np.int32)
    phys = np.zeros(1, dtype=np.int64)
    slot = np.zeros(1, dtype=np.int32)
    st = lib().orc_locate(_p(bt_row), len(bt_row), t, bs, num_blocks, _p(phys), _p(slot))
    return int(st), int(phys[0]), int(slot[0])


class PoolImage:
    """The oracle's own model of the pool bytes (same documented layout)."""

    def __init__(self, num_blocks, block_size, L, H_KV, d_h, elem_bytes, fill: int = 0):
        """elem_bytes: 2 (bf16), 1 (e4m3) or 'int4' (two elements per byte)."""
        self.kind = kind_of(elem_bytes)
        self.N, self.bs, self.L, self.H_KV, self.d_h = num_blocks, block_size, L, H_KV, d_h
        self.s = 2 if self.kind == KIND_BF16 else 1             # bytes per element in logical lists
        elems = L * num_blocks * 2 * H_KV * block_size * d_h
        self.bytes = np.full(elems // 2 if self.kind == KIND_INT4 else elems * self.s, fill, dtype=np.uint8)
        self.scales = np.ones((L, 2, H_KV, d_h), dtype=np.float32)   # e4m3 pools only

    def layer_view(self, layer: int) -> np.ndarray:
        n = self.bytes.size // self.L
        return self.bytes[layer * n:(layer + 1) * n]

    def offset(self, layer, phys, kv, h, slot, c) -> int:
        return int(lib().orc_pool_offset(self.N, self.bs, self.H_KV, self.d_h, layer, phys, kv, h, slot, c))

    def write_tokens(self, layer, block_tables, start_pos, cu, k_bits, v_bits) -> int:
        bt = np.ascontiguousarray(block_tables, dtype=np.int32)
        B, mb = bt.shape
        sp = np.ascontiguousarray(start_pos, dtype=np.int32)
        cu = np.ascontiguousarray(cu, dtype=np.int64)
        k = np.ascontiguousarray(k_bits, dtype=np.uint16)
        v = np.ascontiguousarray(v_bits, dtype=np.uint16)
        sc = np.ascontiguousarray(self.scales[layer])
        return int(lib().orc_write_tokens(_p(self.bytes), self.N, self.bs, self.H_KV, self.d_h, self.kind,
                                          layer, _p(bt), mb, B, _p(sp), _p(cu), _p(k), _p(v), _p(sc)))

    def append(self, layer, block_tables, lens_pre, k_new, v_new) -> int:
        """Eq. 21.6 for every sequence: one token at position lens_pre[b]."""
        B = len(lens_pre)
        cu = np.arange(B + 1, dtype=np.int64)
        return self.write_tokens(layer, block_tables, lens_pre, cu,
                                 np.asarray(k_new).reshape(B, self.H_KV, self.d_h),
                                 np.asarray(v_new).reshape(B, self.H_KV, self.d_h))

    def gather(self, layer, bt_row, length):
        """Stored scalars of one sequence read back through its table."""
        bt_row = np.ascontiguousarray(bt_row, dtype=np.int32)
        dt = np.uint16 if self.s == 2 else np.uint8
        k = np.empty((length, self.H_KV, self.d_h), dtype=dt)
        v = np.empty_like(k)
        st = lib().orc_gather(_p(self.bytes), self.N, self.bs, self.H_KV, self.d_h, self.kind, layer,
                              _p(bt_row), len(bt_row), length, _p(k), _p(v))
        return int(st), k, v


# ------------------------------------------------------------------ attention
def decode(q_bits, K, V, cu, n, H_KV, scales=None, scale=None, kind=None):
    """Decode attention over logical lists.

    q_bits: bf16 [B][H_Q][d_h]; K, V: stored scalars (uint16 bf16 or uint8 e4m3)
    [total][H_KV][d_h]; cu: int64 [B+1] row offsets; n: int64 [B] positions
    attended; scales: fp32 [2][H_KV][d_h] for e4m3.  Returns (out [B][H_Q][d_h]
    float64, lse [B][H_Q] float64)."""
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    B, H_Q, d = q.shape
    K = np.ascontiguousarray(K)
    V = np.ascontiguousarray(V)
    kind = kind_of(kind if kind is not None else K.dtype.itemsize)
    cu = np.ascontiguousarray(cu, dtype=np.int64)
    n = np.ascontiguousarray(n, dtype=np.int64)
    sc = None if scales is None else np.ascontiguousarray(scales, dtype=np.float32)
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(d)))
    out = np.empty((B, H_Q, d), dtype=np.float64)
    lse = np.empty((B, H_Q), dtype=np.float64)
    st = lib().orc_decode(_p(q), _p(K), _p(V), _p(cu), _p(n), B, H_Q, H_KV, d, kind, _p(sc),
                          float(scale), _p(out), _p(lse))
    if st != OK:
        raise ValueError(f"oracle decode status {st}")
    return out, lse


def prefill(q_bits, K, V, q_start, H_KV, scales=None, scale=None, kind=None):
    """Causal chunk: query i (position q_start+i) reads positions 0..q_start+i of K/V [len][H_KV][d_h]."""
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    n_q, H_Q, d = q.shape
    K = np.ascontiguousarray(K)
    V = np.ascontiguousarray(V)
    assert K.shape[0] >= q_start + n_q
    sc = None if scales is None else np.ascontiguousarray(scales, dtype=np.float32)
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(d)))
    out = np.empty((n_q, H_Q, d), dtype=np.float64)
    lse = np.empty((n_q, H_Q), dtype=np.float64)
    st = lib().orc_prefill(_p(q), n_q, _p(K), _p(V), q_start, H_Q, H_KV, d,
                           kind_of(kind if kind is not None else K.dtype.itemsize), _p(sc),
                           float(scale), _p(out), _p(lse))
    if st != OK:
        raise ValueError(f"oracle prefill status {st}")
    return out, lse


def timed(fn, *a, **kw):
    t0 = time.perf_counter()
    r = fn(*a, **kw)
    return r, time.perf_counter() - t0
