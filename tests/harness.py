"""Drive one workload through the CUDA library (C ABI) and through the oracle.

Both sides consume the same generated host arrays (``synth``); neither sees
the other's results.  Used by the GPU tests, ``__graft_entry__.smoke()`` and
``bench.py``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch

import synth
from synth.workloads import K_KIND, V_KIND, Workload

# tolerances on attention outputs (fp32 accumulation on the GPU vs fp64 oracle)
TOL_OUT = {"bf16": 1e-2, "fp8": 3e-2, "int4": 3e-2}
TOL_LSE_REL = 2e-3


@dataclass
class LayerData:
    """Host inputs of one layer: context write units, the step's q / new K,V."""
    k_ctx: np.ndarray          # bf16 bits [T][H_KV][d_h], write units concatenated
    v_ctx: np.ndarray
    cu: np.ndarray             # int32 [U+1]
    start: np.ndarray          # int32 [U] first position of each unit
    rows: np.ndarray           # int32 [U] table row of each unit
    q: np.ndarray              # bf16 bits [B][H_Q][d_h]
    k_new: np.ndarray          # bf16 bits [B][H_KV][d_h]
    v_new: np.ndarray


def layer_data(w: Workload, layer: int, with_step: bool = True) -> LayerData:
    units = []                 # (row, start, end)
    if w.shared_prefix:
        units.append((0, 0, w.shared_prefix))
    for b in range(w.B):
        units.append((b, w.shared_prefix, int(w.lens_pre[b])))
    ks, vs, cu = [], [], [0]
    for (r, s, e) in units:
        ks.append(w.ctx_tokens(layer, K_KIND, r, s, e))
        vs.append(w.ctx_tokens(layer, V_KIND, r, s, e))
        cu.append(cu[-1] + (e - s))
    shape = (0, w.H_KV, w.d_h)
    return LayerData(
        k_ctx=np.concatenate(ks) if ks else np.zeros(shape, np.uint16),
        v_ctx=np.concatenate(vs) if vs else np.zeros(shape, np.uint16),
        cu=np.array(cu, dtype=np.int32), start=np.array([u[1] for u in units], dtype=np.int32),
        rows=np.array([u[0] for u in units], dtype=np.int32),
        q=w.q(layer) if with_step else None,
        k_new=w.kv_new(layer, K_KIND) if with_step else None,
        v_new=w.kv_new(layer, V_KIND) if with_step else None)


def logical_lists(w: Workload, ld: LayerData, stored_k: np.ndarray, stored_v: np.ndarray,
                  new_k: np.ndarray, new_v: np.ndarray):
    """Per-sequence logical lists [sum(len_pre+1)][H_KV][d_h] of stored scalars:
    the context (shared prefix first) followed by the appended token."""
    sp = w.shared_prefix
    parts_k, parts_v, cu = [], [], [0]
    u0 = 1 if sp else 0
    for b in range(w.B):
        a, e = int(ld.cu[u0 + b]), int(ld.cu[u0 + b + 1])
        if sp:
            parts_k.append(stored_k[:sp])
            parts_v.append(stored_v[:sp])
        parts_k += [stored_k[a:e], new_k[b:b + 1]]
        parts_v += [stored_v[a:e], new_v[b:b + 1]]
        cu.append(cu[-1] + sp + (e - a) + 1)
    return np.concatenate(parts_k), np.concatenate(parts_v), np.array(cu, dtype=np.int64)


# ---------------------------------------------------------------- torch helpers
def dev_bits(bits: np.ndarray, device="cuda") -> torch.Tensor:
    """uint16 bf16 bit patterns -> CUDA bfloat16 tensor (bit for bit)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def dev_i32(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)


# ---------------------------------------------------------------- GPU side
class GpuCase:
    """A workload's pool on the GPU, filled through kvc_write_tokens."""

    def __init__(self, kvc, w: Workload, fill_byte: int = 0xFF, device="cuda"):
        self.kvc, self.w, self.device = kvc, w, device
        dt = {"bf16": kvc.KVC_BF16, "fp8": kvc.KVC_FP8_E4M3, "int4": kvc.KVC_INT4}[w.dtype]
        self.pool = kvc.kvc_pool_create(w.num_blocks, w.bs, w.L, w.H_KV, w.d_h, dt)
        self.pool.bytes_view().fill_(fill_byte)
        self.bt = dev_i32(w.block_tables, device)
        self.bt_dec = self.bt[:w.B].contiguous()
        self.lens_pre = dev_i32(w.lens_pre, device)
        self.lens_post = dev_i32(w.lens_post, device)

    def load_context(self, layer: int, ld: LayerData, calibrate: bool = True):
        kvc, w = self.kvc, self.w
        if len(ld.k_ctx) == 0:
            return
        k, v = dev_bits(ld.k_ctx, self.device), dev_bits(ld.v_ctx, self.device)
        if w.dtype != "bf16" and calibrate:
            kvc.kvc_calibrate_scales(self.pool, layer, k, v)
        unit_bt = dev_i32(w.block_tables[ld.rows], self.device)
        max_tok = int(np.max(ld.cu[1:] - ld.cu[:-1]))
        kvc.kvc_write_tokens(self.pool, layer, unit_bt, dev_i32(ld.start, self.device),
                             dev_i32(ld.cu, self.device), k, v, max_tokens=max_tok)
        del k, v

    def step_inputs(self, ld: LayerData):
        return dev_bits(ld.q, self.device), dev_bits(ld.k_new, self.device), dev_bits(ld.v_new, self.device)

    def step(self, layer: int, ld: LayerData, q=None, k_new=None, v_new=None, out=None, lse=None):
        """Append (Eq. 21.6) then decode attention; returns (out, lse) on the device."""
        kvc, w = self.kvc, self.w
        if q is None:
            q, k_new, v_new = self.step_inputs(ld)
        if out is None:
            out = torch.empty((w.B, w.H_Q, w.d_h), dtype=torch.float32, device=self.device)
            lse = torch.empty((w.B, w.H_Q), dtype=torch.float32, device=self.device)
        kvc.kvc_append(self.pool, layer, self.bt_dec, self.lens_pre, k_new, v_new)
        kvc.kvc_decode_attn(self.pool, layer, q, self.bt_dec, self.lens_post, out, lse, scale=w.scale)
        return out, lse

    def layer_bytes(self, layer: int) -> np.ndarray:
        view = self.pool.bytes_view()
        n = view.numel() // self.w.L
        return view[layer * n:(layer + 1) * n].cpu().numpy()

    def close(self):
        self.pool.close()


# ---------------------------------------------------------------- oracle side
class OracleCase:
    """The oracle's image of one layer and its decode result."""

    def __init__(self, w: Workload, fill_byte: int = 0xFF):
        import oracle
        self.oracle, self.w = oracle, w
        self.fill = fill_byte

    def run_layer(self, ld: LayerData, decode: bool = True, image: bool = True):
        o, w = self.oracle, self.w
        s = {"bf16": 2, "fp8": 1, "int4": "int4"}[w.dtype]
        scales = None
        if w.dtype == "fp8":
            scales = np.stack([o.fp8_scales(ld.k_ctx), o.fp8_scales(ld.v_ctx)]).astype(np.float32)
        elif w.dtype == "int4":
            scales = np.stack([o.int4_scales(ld.k_ctx), o.int4_scales(ld.v_ctx)]).astype(np.float32)
        img = None
        if image:
            img = o.PoolImage(w.num_blocks, w.bs, 1, w.H_KV, w.d_h, s, fill=self.fill)
            if scales is not None:
                img.scales[0] = scales
            st = img.write_tokens(0, w.block_tables[ld.rows], ld.start, ld.cu.astype(np.int64), ld.k_ctx, ld.v_ctx)
            assert st == o.OK, st
            st = img.append(0, w.block_tables[:w.B], w.lens_pre, ld.k_new, ld.v_new)
            assert st == o.OK, st
        res = {"image": img, "scales": scales}
        if decode:
            if scales is None:
                sk, sv, nk, nv = ld.k_ctx, ld.v_ctx, ld.k_new, ld.v_new
            else:
                qz = o.quantize_e4m3 if w.dtype == "fp8" else o.quantize_int4
                sk, sv = qz(ld.k_ctx, scales[0]), qz(ld.v_ctx, scales[1])
                nk, nv = qz(ld.k_new, scales[0]), qz(ld.v_new, scales[1])
            K, V, cu = logical_lists(w, ld, sk, sv, nk, nv)
            out, lse = o.decode(ld.q, K, V, cu, w.lens_post.astype(np.int64), w.H_KV, scales=scales, scale=w.scale,
                                kind=w.dtype)
            res.update(out=out, lse=lse, K=K, V=V, cu=cu)
        return res


def check_attention(out_gpu, lse_gpu, out_ref, lse_ref, dtype: str, what: str = ""):
    """Tolerance check; returns (max |out err|, max scaled lse err)."""
    o = out_gpu.detach().cpu().numpy().astype(np.float64) if isinstance(out_gpu, torch.Tensor) else out_gpu
    l = lse_gpu.detach().cpu().numpy().astype(np.float64) if isinstance(lse_gpu, torch.Tensor) else lse_gpu
    assert np.all(np.isfinite(o)), f"{what}: non-finite outputs"
    err_o = float(np.max(np.abs(o - out_ref))) if o.size else 0.0
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(l), fin), f"{what}: lse finiteness differs"
    err_l = float(np.max(np.abs(l[fin] - lse_ref[fin]) / np.maximum(1.0, np.abs(lse_ref[fin])))) if fin.any() else 0.0
    assert err_o <= TOL_OUT[dtype], f"{what}: max |out - ref| = {err_o:.3e} > {TOL_OUT[dtype]}"
    assert err_l <= TOL_LSE_REL, f"{what}: lse error {err_l:.3e} > {TOL_LSE_REL}"
    return err_o, err_l


def first_mismatch(a: np.ndarray, b: np.ndarray):
    d = np.flatnonzero(a != b)
    return (int(d.size), int(d[0])) if d.size else (0, -1)


def scale_of(d_h: int) -> float:
    return float(np.float32(1.0 / math.sqrt(d_h)))
