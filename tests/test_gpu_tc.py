"""The tensor-memory (tcgen05) kernels against the oracle, through the C ABI.

MQA decode (32 query heads per KV head, bf16 and e4m3, d_h 128) and the prefill chunk
(bf16, d_h 64 / 128, every group size) run on tensor-memory kernels; every
case here also runs with KVC_TC=0 (the warp-level kernels) so both paths are
held to the same oracle.  Shapes start small (one sequence of two blocks, one
query) and grow: partial last tiles (value rows past the end zeroed over
NaN-filled memory), many splits and one split, the fused append, empty
sequences and bad table entries, chunks starting inside a block.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from harness import GpuCase, OracleCase, check_attention, dev_bits, dev_i32, first_mismatch, layer_data

pytestmark = pytest.mark.gpu


def _case(kvc, w, fused: bool, env: dict | None = None, fill=0xFF):
    """One decode step (fused or append + attention) on the GPU and in the oracle."""
    env = env or {}
    saved = {k: os.environ.get(k) for k in env}
    os.environ.update(env)
    g = GpuCase(kvc, w, fill_byte=fill)
    try:
        ld = layer_data(w, 0)
        g.load_context(0, ld)
        q, k_new, v_new = g.step_inputs(ld)
        out = torch.full((w.B, w.H_Q, w.d_h), float("nan"), device="cuda")
        lse = torch.full((w.B, w.H_Q), float("nan"), device="cuda")
        if fused:
            kvc.kvc_decode_step(g.pool, 0, q, g.bt_dec, g.lens_pre, k_new, v_new, out, lse, scale=w.scale)
        else:
            g.step(0, ld, q, k_new, v_new, out, lse)
        torch.cuda.synchronize()
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
        ref = OracleCase(w, fill_byte=fill).run_layer(ld)
        n, first = first_mismatch(g.layer_bytes(0), ref["image"].bytes)
        assert n == 0, f"{n} pool bytes differ, first at {first}"
        err = check_attention(out, lse, ref["out"], ref["lse"], w.dtype, f"{w.name} fused={fused} {env}")
        return out.cpu(), lse.cpu(), err
    finally:
        g.close()
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


MQA_LENS = [[20], [127], [128], [129], [5, 300, 1000], [4000, 1, 2500, 17], [8192, 8192, 3000, 12000]]


@pytest.mark.parametrize("lens", MQA_LENS, ids=[f"B{len(x)}_max{max(x)}" for x in MQA_LENS])
@pytest.mark.parametrize("fused", [False, True], ids=["append_then_attend", "fused_step"])
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_mqa_tensor_memory_decode(kvc, lens, fused, dtype):
    w = synth.make_workload("custom", B=len(lens), H_Q=32, H_KV=1, d_h=128, lens=lens, dtype=dtype,
                            seed=sum(lens) % 97)
    _, _, (err_tc, _) = _case(kvc, w, fused)
    _, _, (err_mma, _) = _case(kvc, w, fused, {"KVC_TC": "0"})
    # the tensor-memory kernels feed ~16-bit weights (high + low parts, bf16 or f16) to the
    # value mixture; the split kernel's 32-head groups feed one part.  On e4m3 pools both
    # kernels round q s_K to f16 (11 bits), the error that dominates, and accumulate the scores
    # in different orders: there the tensor-memory kernel is held to 1.5x the split kernel's
    # error (both stay ~100x inside the e4m3 tolerance)
    assert err_tc <= max(2e-4, (1.5 if dtype == "fp8" else 1.0) * err_mma), (err_tc, err_mma)


@pytest.mark.parametrize("chunk", ["8", "16", "24", "4096", "5", "12", "100"])
@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_mqa_tensor_memory_split_sizes(kvc, chunk, dtype):
    """One tile per split up to one split per sequence (partials merged or not).  The e4m3 kernel takes
    splits that are not whole tiles (5, 12, 100 blocks: the last tile is partial, its blocks past the split
    belong to the next one); for the bf16 kernel they are rounded up to whole tiles."""
    w = synth.make_workload("custom", B=3, H_Q=32, H_KV=1, d_h=128, lens=[3000, 129, 700], dtype=dtype, seed=5)
    _case(kvc, w, True, {"KVC_SPLIT_CHUNK": chunk})


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_mqa_tensor_memory_several_kv_heads(kvc, dtype):
    """H_Q = 64 over 2 KV heads: 32-head groups, grid over (split, KV head, sequence)."""
    w = synth.make_workload("custom", B=2, H_Q=64, H_KV=2, d_h=128, lens=[1500, 260], dtype=dtype, seed=9)
    _case(kvc, w, True)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_mqa_tensor_memory_empty_and_bad_entries(kvc, dtype):
    """An empty sequence gives 0 / -inf; a table entry outside the pool is skipped
    and reported, and the pool stays usable."""
    w = synth.make_workload("custom", B=3, H_Q=32, H_KV=1, d_h=128, lens=[0, 300, 40], dtype=dtype, seed=13,
                            spare_blocks=2)
    g = GpuCase(kvc, w, fill_byte=0)
    try:
        ld = layer_data(w, 0)
        g.load_context(0, ld)
        q, k, v = g.step_inputs(ld)
        lens_post = dev_i32([0, 301, 41])
        out = torch.full((3, 32, 128), float("nan"), device="cuda")
        lse = torch.full((3, 32), float("nan"), device="cuda")
        kvc.kvc_append(g.pool, 0, g.bt_dec[1:], g.lens_pre[1:], k[1:], v[1:])
        kvc.kvc_decode_attn(g.pool, 0, q, g.bt_dec, lens_post, out, lse, scale=w.scale)
        torch.cuda.synchronize()
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
        assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
        assert torch.all(torch.isfinite(out[1:]))
        bad = w.block_tables[:w.B].copy()
        bad[1, 5] = w.num_blocks + 3
        kvc.kvc_decode_attn(g.pool, 0, q, dev_i32(bad), lens_post, out, lse, scale=w.scale)
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_ERR_BAD_BLOCK
        kvc.kvc_decode_attn(g.pool, 0, q, g.bt_dec, lens_post, out, lse, scale=w.scale)
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
        assert torch.all(torch.isfinite(out[1:]))
    finally:
        g.close()


# (q_start, n_q): one query, a chunk inside the first block, a chunk starting inside a
# block, partial query tiles, several 64-key stages, a long chunk over a long prefix
PREFILL_CHUNKS = [(0, 1), (0, 5), (7, 9), (45, 23), (200, 61), (1, 130), (333, 200), (1200, 600)]


def _prefill_case(kvc, H_KV, d_h, q_start, n_q, env=None):
    H_Q = 32
    w = synth.make_workload("custom", B=1, H_Q=H_Q, H_KV=H_KV, d_h=d_h, lens=[q_start + n_q], seed=q_start + n_q + H_KV)
    ld = layer_data(w, 0, with_step=False)
    saved = {k: os.environ.get(k) for k in (env or {})}
    os.environ.update(env or {})
    g = GpuCase(kvc, w, fill_byte=0xFF)
    try:
        g.load_context(0, ld)
        qc = synth.normal_bf16(17, n_q, n_q * H_Q * d_h).reshape(n_q, H_Q, d_h)
        out = torch.full((n_q, H_Q, d_h), float("nan"), device="cuda")
        lse = torch.full((n_q, H_Q), float("nan"), device="cuda")
        kvc.kvc_prefill_attn(g.pool, 0, dev_bits(qc), g.bt[0], q_start, out, lse, scale=w.scale)
        torch.cuda.synchronize()
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
        ro, rl = oracle.prefill(qc, ld.k_ctx, ld.v_ctx, q_start, H_KV, scale=w.scale)
        return check_attention(out, lse, ro, rl, "bf16", f"tc prefill H_KV={H_KV} d_h={d_h} {q_start}+{n_q} {env}")
    finally:
        g.close()
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v


@pytest.mark.parametrize("chunk", PREFILL_CHUNKS, ids=[f"{a}+{b}" for a, b in PREFILL_CHUNKS])
@pytest.mark.parametrize("H_KV,d_h", [(8, 128), (32, 128), (1, 128), (16, 64), (4, 64)])
def test_tensor_memory_prefill(kvc, H_KV, d_h, chunk):
    """Groups of 4, 1 (MHA), 32 (MQA), 2 and 8 query heads per tile of 128 rows,
    head widths 128 and 64, NaN in every unused pool byte; against the oracle,
    and no less accurate than the warp-level prefill kernels (KVC_TC=0)."""
    q_start, n_q = chunk
    err_tc, _ = _prefill_case(kvc, H_KV, d_h, q_start, n_q)
    err_ref, _ = _prefill_case(kvc, H_KV, d_h, q_start, n_q, {"KVC_TC": "0"})
    assert err_tc <= max(4e-3, 2 * err_ref), (err_tc, err_ref)
