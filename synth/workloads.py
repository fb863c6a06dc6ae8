"""Workload recipes: lengths, block tables and the streams that hold each tensor.

Shapes follow the pages' worked examples: the Llama-3.1-8B-style head shape
(32 query heads, 8 KV heads, width 128, bf16) from "KV Cache Explained: The
Memory Problem Behind Fast LLM Inference" ("How much GPU memory does the KV
cache use?"), 16-token blocks from its "Why PagedAttention allocates KV in
blocks", the 1 800-token request with a 1 200-token (75-block) shared prefix
from the xf_kv_cache page's "End-to-end flow".

Every value is N(0,1) rounded to bf16, drawn from a counter-based stream, so a
slice of any tensor (one sequence, a token range) is regenerated on its own.
Physical block ids come from a seeded Fisher-Yates permutation of the pool,
handed out in sequence order; table entries past a sequence's last block are -1.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

from . import normal_bf16, permutation, stream_id, u64, uniform_f64

# stream tags
_CTX, _Q, _NEW, _SHARED, _PREFILL_Q, _LENS, _PERM = 1, 2, 3, 4, 5, 10, 11
K_KIND, V_KIND = 0, 1


@dataclass
class Prefill:
    seq: int            # row of block_tables used by the chunk
    q_start: int        # position of the chunk's first query
    n_q: int            # chunk length
    total: int          # q_start + n_q tokens after the chunk is written


@dataclass
class Workload:
    name: str
    seed: int
    B: int              # decode sequences
    H_Q: int
    H_KV: int
    d_h: int
    bs: int
    L: int
    dtype: str          # "bf16" | "fp8"
    num_blocks: int
    lens_pre: np.ndarray            # int32 [B] cached tokens before the append
    block_tables: np.ndarray        # int32 [rows][max_blocks]; rows = B (+1 with a prefill chunk)
    shared_prefix: int = 0          # leading positions shared by every row (same physical blocks)
    prefill: Optional[Prefill] = None
    notes: dict = field(default_factory=dict)

    # ------------------------------------------------------------ geometry
    @property
    def g(self) -> int:
        return self.H_Q // self.H_KV

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def elem_bits(self) -> int:
        return {"bf16": 16, "fp8": 8, "int4": 4}[self.dtype]

    @property
    def elem_bytes(self) -> float:
        return self.elem_bits / 8

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(d_h), as the fp32 value passed to the kernels."""
        return float(np.float32(1.0 / math.sqrt(self.d_h)))

    @property
    def lens_post(self) -> np.ndarray:
        return (self.lens_pre + 1).astype(np.int32)

    def row_len(self, b: int) -> int:
        """Tokens held by row b before the step (the prefill row holds its whole chunk)."""
        if self.prefill is not None and b == self.prefill.seq:
            return self.prefill.total
        return int(self.lens_pre[b])

    # ------------------------------------------------------------ values
    def ctx_tokens(self, layer: int, kind: int, b: int, t0: int, t1: int) -> np.ndarray:
        """bf16 bits [t1-t0][H_KV][d_h] of row b's cached keys (kind 0) or values (kind 1)."""
        row = self.H_KV * self.d_h
        out = np.empty((t1 - t0, self.H_KV, self.d_h), dtype=np.uint16)
        flat = out.reshape(-1)
        s = min(max(self.shared_prefix, t0), t1)
        if s > t0:   # shared prefix: one stream for every row
            flat[: (s - t0) * row] = normal_bf16(
                self.seed, stream_id(_SHARED, layer, kind), (s - t0) * row, offset=t0 * row)
        if t1 > s:
            flat[(s - t0) * row:] = normal_bf16(
                self.seed, stream_id(_CTX, layer, kind, b), (t1 - s) * row, offset=s * row)
        return out

    def q(self, layer: int) -> np.ndarray:
        """bf16 bits [B][H_Q][d_h]: the step's queries."""
        n = self.B * self.H_Q * self.d_h
        return normal_bf16(self.seed, stream_id(_Q, layer), n).reshape(self.B, self.H_Q, self.d_h)

    def kv_new(self, layer: int, kind: int) -> np.ndarray:
        """bf16 bits [B][H_KV][d_h]: the step's new key (kind 0) or value (kind 1)."""
        n = self.B * self.H_KV * self.d_h
        return normal_bf16(self.seed, stream_id(_NEW, layer, kind), n).reshape(self.B, self.H_KV, self.d_h)

    def prefill_q(self, layer: int) -> np.ndarray:
        p = self.prefill
        n = p.n_q * self.H_Q * self.d_h
        return normal_bf16(self.seed, stream_id(_PREFILL_Q, layer), n).reshape(p.n_q, self.H_Q, self.d_h)

    # ------------------------------------------------------------ bytes
    def kv_bytes_read(self) -> int:
        """Valid cached K+V bytes one decode-attention pass reads per layer."""
        return int(self.lens_post.astype(np.int64).sum()) * 2 * self.H_KV * self.d_h * self.elem_bits // 8


def _tables(lens_need: np.ndarray, perm: np.ndarray, bs: int, max_blocks: int,
            shared_blocks: int = 0) -> np.ndarray:
    """Hand out physical blocks in sequence order from a permutation.

    ``lens_need[r]`` tokens must fit row r.  The first ``shared_blocks`` ids of
    the permutation are mapped into every row's leading entries."""
    rows = len(lens_need)
    bt = np.full((rows, max_blocks), -1, dtype=np.int32)
    cur = shared_blocks
    for r in range(rows):
        nb = -(-int(lens_need[r]) // bs)
        bt[r, :shared_blocks] = perm[:shared_blocks]
        own = nb - shared_blocks
        bt[r, shared_blocks:nb] = perm[cur:cur + own]
        cur += own
    assert cur <= len(perm), "pool too small for the tables"
    return bt


def make_workload(name: str, seed: int = 0, **kw) -> Workload:
    """Build one of the named workloads (see WORKLOADS) or a custom one.

    Custom keyword form: B, H_Q, H_KV, d_h, lens (list or int), L=1, bs=16,
    dtype='bf16', spare_blocks=0."""
    if name == "tiny":          # 4 sequences, lengths U[1,256], 128-block pool
        B, H_Q, H_KV, d, bs, L, N = 4, 8, 2, 64, 16, 1, 128
        lens = (1 + (u64(seed, stream_id(_LENS), B) % np.uint64(256))).astype(np.int32)
        perm = permutation(seed, stream_id(_PERM), N)
        mb = -(-(int(lens.max()) + 1) // bs)
        bt = _tables(lens + 1, perm, bs, mb)
        return Workload(name, seed, B, H_Q, H_KV, d, bs, L, "bf16", N, lens, bt)

    if name == "llama_gqa":     # B=32, context 8192, one layer
        return _uniform(name, seed, B=32, H_Q=32, H_KV=8, d=128, ctx=8192, L=1, dtype="bf16")

    if name.startswith("sweep_"):   # sweep_hkv{32,8,1}_{bf16,fp8,int4}: B=8, context 32768
        _, hk, dt = name.split("_")
        return _uniform(name, seed, B=8, H_Q=32, H_KV=int(hk[3:]), d=128, ctx=32768, L=1, dtype=dt)

    if name == "full_pool":     # 32 layers, 8 x 32768 tokens = 32 GiB, +8 blocks for the append
        return _uniform(name, seed, B=8, H_Q=32, H_KV=8, d=128, ctx=32768, L=32, dtype="bf16")

    if name == "ragged_prefix":  # 64 log-uniform lengths, 1200-token shared prefix + 600-token chunk
        return _ragged_prefix(seed, **kw)

    if name == "custom":
        B, H_Q, H_KV, d = kw["B"], kw["H_Q"], kw["H_KV"], kw["d_h"]
        bs, L, dt = kw.get("bs", 16), kw.get("L", 1), kw.get("dtype", "bf16")
        lens = kw["lens"]
        lens = np.full(B, lens, dtype=np.int32) if np.isscalar(lens) else np.asarray(lens, dtype=np.int32)
        need = lens + 1
        nb = -(-need // bs)
        N = int(nb.sum()) + int(kw.get("spare_blocks", 0))
        perm = permutation(seed, stream_id(_PERM), N)
        mb = max(1, int(nb.max()) + int(kw.get("extra_cols", 0))) if B else 1
        bt = _tables(need, perm, bs, mb)
        return Workload(kw.get("label", "custom"), seed, B, H_Q, H_KV, d, bs, L, dt, N, lens, bt)

    raise KeyError(name)


def _uniform(name, seed, B, H_Q, H_KV, d, ctx, L, dtype) -> Workload:
    bs = 16
    lens = np.full(B, ctx, dtype=np.int32)
    nb = -(-(ctx + 1) // bs)
    N = B * nb
    perm = permutation(seed, stream_id(_PERM), N)
    bt = _tables(lens + 1, perm, bs, nb)
    return Workload(name, seed, B, H_Q, H_KV, d, bs, L, dtype, N, lens, bt)


def _ragged_prefix(seed, B=64, shared=1200, chunk=600, lo=128, hi=32768, H_Q=32, H_KV=8, dtype="bf16") -> Workload:
    bs = 16
    assert shared % bs == 0, "the shared prefix fills whole blocks"
    u = uniform_f64(seed, stream_id(_LENS), B)
    raw = np.rint(np.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))).astype(np.int64)
    lens = np.maximum(raw, shared).astype(np.int32)
    sb = shared // bs
    total = shared + chunk
    need = np.concatenate([lens + 1, [total]]).astype(np.int64)
    nb = -(-need // bs)
    N = sb + int((nb - sb).sum())
    perm = permutation(seed, stream_id(_PERM), N)
    bt = _tables(need, perm, bs, int(nb.max()), shared_blocks=sb)
    w = Workload("ragged_prefix", seed, B, H_Q, H_KV, 128, bs, 1, dtype, N, lens, bt,
                 shared_prefix=shared, prefill=Prefill(seq=B, q_start=shared, n_q=chunk, total=total))
    w.notes["clamped_to_prefix"] = int((raw < shared).sum())
    return w


WORKLOADS = ["tiny", "llama_gqa", "ragged_prefix",
             "sweep_hkv32_bf16", "sweep_hkv8_bf16", "sweep_hkv1_bf16",
             "sweep_hkv32_fp8", "sweep_hkv8_fp8", "sweep_hkv1_fp8", "full_pool",
             "sweep_hkv32_int4", "sweep_hkv8_int4", "sweep_hkv1_int4"]
