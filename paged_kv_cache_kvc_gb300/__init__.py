"""Python binding of libkvc: a paged KV cache and its decode step on GB300.

Argument marshalling only: every step runs in the CUDA library's kernels
(``csrc/``), reached through its C ABI (``include/kvc.h``) with ctypes.
PyTorch supplies device memory and streams.  The names match the C entry
points; tensors are passed where the C call takes device pointers, and the
stream defaults to torch's current stream.

There is no fallback: if the library is not built, ``load()`` raises.  Build
it with ``python -c "import __graft_entry__ as g; g.build()"`` (or
``paged_kv_cache_kvc_gb300/build.py``).
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libkvc.so")

KVC_BF16, KVC_FP8_E4M3, KVC_INT4 = 0, 1, 2
(KVC_OK, KVC_ERR_ARG, KVC_ERR_OOM, KVC_ERR_BAD_BLOCK, KVC_ERR_RANGE, KVC_ERR_ALIAS, KVC_ERR_STALE,
 KVC_ERR_TIMEOUT, KVC_ERR_CUDA, KVC_ERR_UNSUPPORTED) = range(10)

_lib = None


class KvcError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {kvc_status_str(status)} (status {status})")


class kvc_pool_desc(ctypes.Structure):
    _fields_ = [("layout_version", ctypes.c_int32), ("block_size", ctypes.c_int32), ("num_layers", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("elem_bytes", ctypes.c_int32), ("device", ctypes.c_int32), ("num_blocks", ctypes.c_int64),
                ("block_bytes_per_layer", ctypes.c_uint64), ("layer_bytes", ctypes.c_uint64),
                ("bytes_per_token", ctypes.c_uint64), ("capacity_tokens", ctypes.c_uint64),
                ("pool_bytes", ctypes.c_uint64), ("base", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("elem_bits", ctypes.c_int32), ("reserved", ctypes.c_int32)]


EXPORTS = ["kvc_pool_create", "kvc_pool_destroy", "kvc_pool_info", "kvc_pool_set_scales", "kvc_calibrate_fp8",
           "kvc_calibrate_scales",
           "kvc_append", "kvc_write_tokens", "kvc_decode_attn", "kvc_prefill_attn", "kvc_pool_reserve",
           "kvc_bytes", "kvc_pool_sync_status", "kvc_status_str", "kvc_launch_count", "kvc_decode_attn_noalloc", "kvc_decode_step",
           "kvc_mixed_step",
           "kvc_alloc_create", "kvc_alloc_destroy", "kvc_alloc_new_seq", "kvc_alloc_fork", "kvc_alloc_reserve",
           "kvc_alloc_commit", "kvc_alloc_release", "kvc_alloc_publish", "kvc_alloc_match", "kvc_alloc_seq_info",
           "kvc_alloc_block_tables", "kvc_alloc_counts", "kvc_alloc_refcount", "kvc_alloc_lease", "kvc_alloc_check",
           "kvc_copy_blocks"]


def load(path: str = LIB_PATH):
    """Load libkvc.so (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libkvc is not built ({path} missing); run __graft_entry__.build()")
    L = ctypes.CDLL(path)
    vp, i32, i64, u64, st = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_int
    f = L.kvc_pool_create
    f.restype, f.argtypes = st, [i64, i32, i32, i32, i32, ctypes.c_int, ctypes.POINTER(vp)]
    L.kvc_pool_destroy.restype, L.kvc_pool_destroy.argtypes = None, [vp]
    L.kvc_pool_info.restype, L.kvc_pool_info.argtypes = st, [vp, ctypes.POINTER(kvc_pool_desc)]
    L.kvc_pool_set_scales.restype, L.kvc_pool_set_scales.argtypes = st, [vp, i32, vp, vp, vp]
    L.kvc_calibrate_fp8.restype, L.kvc_calibrate_fp8.argtypes = st, [vp, i32, vp, vp, i64, i32, vp]
    L.kvc_calibrate_scales.restype, L.kvc_calibrate_scales.argtypes = st, [vp, i32, vp, vp, i64, i32, vp]
    L.kvc_append.restype, L.kvc_append.argtypes = st, [vp, i32, vp, i32, vp, i32, vp, vp, vp]
    L.kvc_write_tokens.restype, L.kvc_write_tokens.argtypes = st, [vp, i32, vp, i32, vp, vp, i32, i32, vp, vp, vp]
    L.kvc_decode_attn.restype = st
    L.kvc_decode_attn.argtypes = [vp, i32, vp, i32, vp, i32, vp, i32, vp, vp, ctypes.c_float, vp]
    L.kvc_decode_step.restype = st
    L.kvc_decode_step.argtypes = [vp, i32, vp, i32, vp, i32, vp, i32, vp, vp, vp, vp, ctypes.c_float, vp]
    L.kvc_decode_attn_noalloc.restype = st
    L.kvc_decode_attn_noalloc.argtypes = [vp, i32, vp, i32, vp, i32, vp, i32, vp, vp, ctypes.c_float, vp]
    L.kvc_prefill_attn.restype = st
    L.kvc_prefill_attn.argtypes = [vp, i32, vp, i32, i32, vp, i32, i32, vp, vp, ctypes.c_float, vp]
    L.kvc_mixed_step.restype = st
    L.kvc_mixed_step.argtypes = [vp, i32, vp, i32, vp, i32, vp, i32, vp, vp, vp, vp,
                                 vp, i32, vp, i32, i32, vp, vp, ctypes.c_float, vp]
    L.kvc_pool_reserve.restype, L.kvc_pool_reserve.argtypes = st, [vp, i32, i32, i32]
    L.kvc_bytes.restype, L.kvc_bytes.argtypes = u64, [i64] * 6
    L.kvc_pool_sync_status.restype, L.kvc_pool_sync_status.argtypes = st, [vp, vp]
    L.kvc_status_str.restype, L.kvc_status_str.argtypes = ctypes.c_char_p, [st]
    L.kvc_launch_count.restype, L.kvc_launch_count.argtypes = u64, []
    L.kvc_alloc_create.restype, L.kvc_alloc_create.argtypes = st, [i64, i32, vp, i32, ctypes.POINTER(vp)]
    L.kvc_alloc_destroy.restype, L.kvc_alloc_destroy.argtypes = None, [vp]
    L.kvc_alloc_new_seq.restype, L.kvc_alloc_new_seq.argtypes = st, [vp, vp]
    L.kvc_alloc_fork.restype, L.kvc_alloc_fork.argtypes = st, [vp, i32, i32, vp]
    L.kvc_alloc_reserve.restype, L.kvc_alloc_reserve.argtypes = st, [vp, i32, i32, vp, i32, vp]
    L.kvc_alloc_commit.restype, L.kvc_alloc_commit.argtypes = st, [vp, i32, i32]
    L.kvc_alloc_release.restype, L.kvc_alloc_release.argtypes = st, [vp, i32]
    L.kvc_alloc_publish.restype, L.kvc_alloc_publish.argtypes = st, [vp, i32, vp, i32, u64]
    L.kvc_alloc_match.restype, L.kvc_alloc_match.argtypes = st, [vp, vp, i32, u64, vp, vp]
    L.kvc_alloc_seq_info.restype, L.kvc_alloc_seq_info.argtypes = st, [vp, i32, vp, vp]
    L.kvc_alloc_block_tables.restype, L.kvc_alloc_block_tables.argtypes = st, [vp, vp, i32, i32, vp, vp]
    L.kvc_alloc_counts.restype, L.kvc_alloc_counts.argtypes = st, [vp, vp, vp, vp]
    L.kvc_alloc_refcount.restype, L.kvc_alloc_refcount.argtypes = i32, [vp, i32]
    L.kvc_alloc_lease.restype, L.kvc_alloc_lease.argtypes = st, [vp, i32, ctypes.POINTER(u64)]
    L.kvc_alloc_check.restype, L.kvc_alloc_check.argtypes = st, [vp, i32, u64]
    L.kvc_copy_blocks.restype, L.kvc_copy_blocks.argtypes = st, [vp, vp, i32, vp]
    _lib = L
    return L


def _check(status: int, where: str):
    if status != KVC_OK:
        raise KvcError(status, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t, dtype=None, name="tensor", optional=False):
    """Device pointer of a contiguous CUDA tensor (None -> NULL when optional)."""
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


class Pool:
    """Owning handle of a kvc_pool (destroyed on close() or garbage collection)."""

    def __init__(self, handle: int):
        self.handle = handle
        d = kvc_pool_info(self)
        self.num_blocks, self.block_size, self.num_layers = d.num_blocks, d.block_size, d.num_layers
        self.num_kv_heads, self.head_dim, self.dtype, self.elem_bytes = d.num_kv_heads, d.head_dim, d.dtype, d.elem_bytes
        self.elem_bits = d.elem_bits
        self.device = d.device

    def close(self):
        if self.handle:
            load().kvc_pool_destroy(ctypes.c_void_p(self.handle))
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def bytes_view(self) -> torch.Tensor:
        """uint8 CUDA tensor aliasing the whole pool (no copy; valid while the pool lives)."""
        d = kvc_pool_info(self)
        return _alias(d.base, d.pool_bytes, torch.uint8, self.device)

    def scales_view(self) -> torch.Tensor:
        """fp32 [L][2][H_KV][d_h] CUDA tensor aliasing the e4m3 scales."""
        d = kvc_pool_info(self)
        if not d.scales:
            raise ValueError("bf16 pools have no scales")
        n = d.num_layers * 2 * d.num_kv_heads * d.head_dim
        return _alias(d.scales, n * 4, torch.float32, self.device).view(d.num_layers, 2, d.num_kv_heads, d.head_dim)


class _CudaArrayInterface:
    def __init__(self, ptr, nbytes):
        self.__cuda_array_interface__ = {"shape": (nbytes,), "typestr": "|u1", "data": (ptr, False), "version": 3,
                                         "strides": None}


def _alias(ptr: int, nbytes: int, dtype, device: int) -> torch.Tensor:
    with torch.cuda.device(device):
        t = torch.as_tensor(_CudaArrayInterface(ptr, nbytes), device=f"cuda:{device}")
    return t.view(dtype)


def _h(pool) -> ctypes.c_void_p:
    return ctypes.c_void_p(pool.handle if isinstance(pool, Pool) else int(pool))


# ---------------------------------------------------------------------- entry points
def kvc_pool_create(num_blocks, block_size, num_layers, num_kv_heads, head_dim, dtype=KVC_BF16) -> Pool:
    out = ctypes.c_void_p()
    _check(load().kvc_pool_create(num_blocks, block_size, num_layers, num_kv_heads, head_dim, dtype,
                                  ctypes.byref(out)), "kvc_pool_create")
    return Pool(out.value)


def kvc_pool_destroy(pool: Pool):
    pool.close()


def kvc_pool_info(pool) -> kvc_pool_desc:
    d = kvc_pool_desc()
    _check(load().kvc_pool_info(_h(pool), ctypes.byref(d)), "kvc_pool_info")
    return d


def kvc_pool_set_scales(pool, layer, s_k, s_v, stream=None):
    _check(load().kvc_pool_set_scales(_h(pool), layer, _dev(s_k, torch.float32, "s_k"), _dev(s_v, torch.float32, "s_v"),
                                      _stream(stream)), "kvc_pool_set_scales")


def kvc_calibrate_scales(pool, layer, k, v, accumulate=False, stream=None):
    """absmax / 448 (e4m3) or / 7 (int4) per (KV head, channel) over bf16 tokens [n][H_KV][d_h]."""
    n = k.shape[0]
    _check(load().kvc_calibrate_scales(_h(pool), layer, _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"), n,
                                       int(bool(accumulate)), _stream(stream)), "kvc_calibrate_scales")


def kvc_calibrate_fp8(pool, layer, k, v, accumulate=False, stream=None):
    n = k.shape[0]
    _check(load().kvc_calibrate_fp8(_h(pool), layer, _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"), n,
                                    int(bool(accumulate)), _stream(stream)), "kvc_calibrate_fp8")


def kvc_append(pool, layer, block_tables, seq_lens, k_new, v_new, stream=None):
    B, mb = block_tables.shape
    _check(load().kvc_append(_h(pool), layer, _dev(block_tables, torch.int32, "block_tables"), mb,
                             _dev(seq_lens, torch.int32, "seq_lens"), B, _dev(k_new, torch.bfloat16, "k_new"),
                             _dev(v_new, torch.bfloat16, "v_new"), _stream(stream)), "kvc_append")


def kvc_write_tokens(pool, layer, block_tables, start_pos, cu_tokens, k, v, max_tokens=None, stream=None):
    B, mb = block_tables.shape
    if max_tokens is None:
        max_tokens = int((cu_tokens[1:] - cu_tokens[:-1]).max().item()) if B else 0
    _check(load().kvc_write_tokens(_h(pool), layer, _dev(block_tables, torch.int32, "block_tables"), mb,
                                   _dev(start_pos, torch.int32, "start_pos"), _dev(cu_tokens, torch.int32, "cu_tokens"),
                                   B, int(max_tokens), _dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
                                   _stream(stream)), "kvc_write_tokens")


def kvc_decode_attn(pool, layer, q, block_tables, seq_lens, out, lse=None, scale=None, stream=None):
    B, H_Q, D = q.shape
    if scale is None:
        scale = D ** -0.5
    _check(load().kvc_decode_attn(_h(pool), layer, _dev(q, torch.bfloat16, "q"), H_Q,
                                  _dev(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
                                  _dev(seq_lens, torch.int32, "seq_lens"), B, _dev(out, torch.float32, "out"),
                                  _dev(lse, torch.float32, "lse", optional=True), float(scale), _stream(stream)),
           "kvc_decode_attn")


def kvc_decode_step(pool, layer, q, block_tables, seq_lens_pre, k_new, v_new, out, lse=None, scale=None,
                    stream=None):
    """Append (at seq_lens_pre[b]) and decode attention (over seq_lens_pre[b] + 1) in one launch."""
    B, H_Q, D = q.shape
    if scale is None:
        scale = D ** -0.5
    _check(load().kvc_decode_step(_h(pool), layer, _dev(q, torch.bfloat16, "q"), H_Q,
                                  _dev(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
                                  _dev(seq_lens_pre, torch.int32, "seq_lens"), B, _dev(k_new, torch.bfloat16, "k_new"),
                                  _dev(v_new, torch.bfloat16, "v_new"), _dev(out, torch.float32, "out"),
                                  _dev(lse, torch.float32, "lse", optional=True), float(scale), _stream(stream)),
           "kvc_decode_step")


def kvc_decode_attn_noalloc(pool, layer, q, block_tables, seq_lens, out, lse=None, scale=None, stream=None):
    """kvc_decode_attn without any device allocation: split partials go to the
    library's fixed 8 MiB per-device array.  For callers that may not allocate
    during a decode step (memory pre-reserved by their own allocator, or loops
    that cannot afford cudaMalloc's device synchronisation).  Calls that overlap
    on one GPU share the array and race; the first call on a device looks up the
    array's address and should precede any stream capture."""
    B, H_Q, D = q.shape
    if scale is None:
        scale = D ** -0.5
    _check(load().kvc_decode_attn_noalloc(_h(pool), layer, _dev(q, torch.bfloat16, "q"), H_Q,
                                          _dev(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
                                          _dev(seq_lens, torch.int32, "seq_lens"), B, _dev(out, torch.float32, "out"),
                                          _dev(lse, torch.float32, "lse", optional=True), float(scale),
                                          _stream(stream)),
           "kvc_decode_attn_noalloc (a split batch needing more than the 8 MiB scratch is rejected)")


def kvc_prefill_attn(pool, layer, q, block_table_row, q_start, out, lse=None, scale=None, stream=None):
    n_q, H_Q, D = q.shape
    if scale is None:
        scale = D ** -0.5
    _check(load().kvc_prefill_attn(_h(pool), layer, _dev(q, torch.bfloat16, "q"), n_q, H_Q,
                                   _dev(block_table_row, torch.int32, "block_table_row"), block_table_row.shape[-1],
                                   int(q_start), _dev(out, torch.float32, "out"),
                                   _dev(lse, torch.float32, "lse", optional=True), float(scale), _stream(stream)),
           "kvc_prefill_attn")


def kvc_mixed_step(pool, layer, q, block_tables, seq_lens_pre, k_new, v_new, out, lse, prefill_q, prefill_block_table_row,
                   q_start, prefill_out, prefill_lse=None, scale=None, stream=None):
    """kvc_decode_step and kvc_prefill_attn in one launch."""
    B, H_Q, D = q.shape
    n_q = prefill_q.shape[0]
    if scale is None:
        scale = D ** -0.5
    _check(load().kvc_mixed_step(_h(pool), layer, _dev(q, torch.bfloat16, "q"), H_Q,
                                 _dev(block_tables, torch.int32, "block_tables"), block_tables.shape[1],
                                 _dev(seq_lens_pre, torch.int32, "seq_lens"), B, _dev(k_new, torch.bfloat16, "k_new"),
                                 _dev(v_new, torch.bfloat16, "v_new"), _dev(out, torch.float32, "out"),
                                 _dev(lse, torch.float32, "lse", optional=True),
                                 _dev(prefill_q, torch.bfloat16, "prefill_q"), n_q,
                                 _dev(prefill_block_table_row, torch.int32, "prefill_block_table_row"),
                                 prefill_block_table_row.shape[-1], int(q_start),
                                 _dev(prefill_out, torch.float32, "prefill_out"),
                                 _dev(prefill_lse, torch.float32, "prefill_lse", optional=True), float(scale),
                                 _stream(stream)),
           "kvc_mixed_step")


def kvc_pool_reserve(pool, max_batch, num_q_heads, max_blocks):
    _check(load().kvc_pool_reserve(_h(pool), max_batch, num_q_heads, max_blocks), "kvc_pool_reserve")


def kvc_bytes(L, B, H_KV, T, d_h, s) -> int:
    return int(load().kvc_bytes(L, B, H_KV, T, d_h, s))


def kvc_pool_sync_status(pool, stream=None) -> int:
    """Device-detected status since the last call (KVC_OK or a KVC_ERR_* code); does not raise."""
    return int(load().kvc_pool_sync_status(_h(pool), _stream(stream)))


def kvc_status_str(status: int) -> str:
    return load().kvc_status_str(int(status)).decode()


def kvc_launch_count() -> int:
    return int(load().kvc_launch_count())


# ---------------------------------------------------------------------- block allocator (host)
class Allocator:
    """Owning handle of a kvc_alloc: the host block allocator (free queue,
    reference counts, copy-on-write, retention, prefix lookup).  Methods map
    one to one onto the kvc_alloc_* calls."""

    def __init__(self, num_blocks, block_size, free_order=None, retain_cached=False):
        import numpy as np
        L = load()
        self._np = np
        self.block_size = block_size
        out = ctypes.c_void_p()
        fo = None if free_order is None else np.ascontiguousarray(free_order, dtype=np.int32)
        _check(L.kvc_alloc_create(num_blocks, block_size, None if fo is None else fo.ctypes.data,
                                  int(bool(retain_cached)), ctypes.byref(out)), "kvc_alloc_create")
        self.handle = out.value

    def close(self):
        if self.handle:
            load().kvc_alloc_destroy(ctypes.c_void_p(self.handle))
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _h(self):
        return ctypes.c_void_p(self.handle)

    def new_seq(self) -> int:
        s = ctypes.c_int32()
        _check(load().kvc_alloc_new_seq(self._h(), ctypes.byref(s)), "kvc_alloc_new_seq")
        return s.value

    def fork(self, src, n_tokens) -> int:
        s = ctypes.c_int32()
        _check(load().kvc_alloc_fork(self._h(), src, n_tokens, ctypes.byref(s)), "kvc_alloc_fork")
        return s.value

    def reserve(self, seq, n_tokens):
        """Returns the copy-on-write pairs [(old, new)] the caller must copy before writing."""
        pairs = (ctypes.c_int32 * 2)()
        n = ctypes.c_int32()
        _check(load().kvc_alloc_reserve(self._h(), seq, n_tokens, pairs, 1, ctypes.byref(n)), "kvc_alloc_reserve")
        return [(pairs[0], pairs[1])] if n.value else []

    def commit(self, seq, n_tokens):
        _check(load().kvc_alloc_commit(self._h(), seq, n_tokens), "kvc_alloc_commit")

    def release(self, seq):
        _check(load().kvc_alloc_release(self._h(), seq), "kvc_alloc_release")

    def publish(self, seq, tokens, salt=0):
        t = self._np.ascontiguousarray(tokens, dtype=self._np.int32)
        _check(load().kvc_alloc_publish(self._h(), seq, t.ctypes.data if t.size else None, t.size, salt),
               "kvc_alloc_publish")

    def match(self, tokens, salt=0):
        """(new sequence id, positions covered by matched full blocks)."""
        t = self._np.ascontiguousarray(tokens, dtype=self._np.int32)
        s, hit = ctypes.c_int32(), ctypes.c_int32()
        _check(load().kvc_alloc_match(self._h(), t.ctypes.data if t.size else None, t.size, salt, ctypes.byref(s),
                                      ctypes.byref(hit)), "kvc_alloc_match")
        return s.value, hit.value

    def seq_info(self, seq):
        ln, nb = ctypes.c_int64(), ctypes.c_int32()
        _check(load().kvc_alloc_seq_info(self._h(), seq, ctypes.byref(ln), ctypes.byref(nb)), "kvc_alloc_seq_info")
        return ln.value, nb.value

    def block_tables(self, seqs, max_blocks):
        np = self._np
        s = np.ascontiguousarray(seqs, dtype=np.int32)
        table = np.empty((len(s), max_blocks), dtype=np.int32)
        lens = np.empty(len(s), dtype=np.int32)
        _check(load().kvc_alloc_block_tables(self._h(), s.ctypes.data, len(s), max_blocks, table.ctypes.data,
                                             lens.ctypes.data), "kvc_alloc_block_tables")
        return table, lens

    def counts(self):
        f, u, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(load().kvc_alloc_counts(self._h(), ctypes.byref(f), ctypes.byref(u), ctypes.byref(c)),
               "kvc_alloc_counts")
        return {"free": f.value, "used": u.value, "cached": c.value}

    def refcount(self, block) -> int:
        return int(load().kvc_alloc_refcount(self._h(), block))

    def lease(self, seq) -> int:
        """Opaque stamp of the sequence's current block table."""
        st = ctypes.c_uint64()
        _check(load().kvc_alloc_lease(self._h(), seq, ctypes.byref(st)), "kvc_alloc_lease")
        return st.value

    def check(self, seq, stamp) -> bool:
        """True while `stamp` is current; False once it is stale (KVC_ERR_STALE)."""
        r = load().kvc_alloc_check(self._h(), seq, int(stamp))
        if r == KVC_ERR_STALE:
            return False
        _check(r, "kvc_alloc_check")
        return True


def kvc_copy_blocks(pool, pairs, stream=None):
    """pairs: CUDA int32 [n][2] (src, dst): copy whole blocks, every layer."""
    n = pairs.shape[0]
    _check(load().kvc_copy_blocks(_h(pool), _dev(pairs, torch.int32, "pairs") if n else None, n, _stream(stream)),
           "kvc_copy_blocks")
