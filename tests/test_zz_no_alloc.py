"""kvc_decode_attn_noalloc: decode attention for callers that may not allocate
device memory during a decode step (memory pre-reserved by their own caching
allocator, or loops that cannot afford cudaMalloc's device synchronisation).

It must give the results of kvc_decode_attn, call after call, while its split
partials live in the library's fixed per-device scratch array, and it must
refuse a split batch whose partials would not fit that array.  Collected last
so that a run stopping at its first failure has run every other test.
"""
import os

import numpy as np
import pytest
import torch

import synth
from harness import TOL_LSE_REL, TOL_OUT, GpuCase, dev_i32, layer_data

pytestmark = pytest.mark.gpu

SCRATCH_FLOATS = 2 << 20     # the array's documented size: 8 MiB


def _close(a_out, a_lse, b_out, b_lse, dtype):
    err_o = (a_out - b_out).abs().max().item()
    fin = torch.isfinite(b_lse)
    assert torch.equal(torch.isfinite(a_lse), fin)
    err_l = ((a_lse[fin] - b_lse[fin]).abs() / b_lse[fin].abs().clamp(min=1.0)).max().item()
    assert err_o <= TOL_OUT[dtype] and err_l <= TOL_LSE_REL, (err_o, err_l)


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
@pytest.mark.parametrize("lens", [[5000, 3000, 17], [700]])
def test_noalloc_matches_decode_attn_twice(kvc, dtype, lens):
    """Two calls in a row (the second with new queries, so stale scratch from the
    first cannot pass for a result) against kvc_decode_attn."""
    w = synth.make_workload("custom", B=len(lens), H_Q=32, H_KV=8, d_h=128, lens=lens, dtype=dtype, seed=3)
    g = GpuCase(kvc, w)
    try:
        ld = layer_data(w, 0)
        g.load_context(0, ld)
        q, k_new, v_new = g.step_inputs(ld)
        kvc.kvc_append(g.pool, 0, g.bt_dec, g.lens_pre, k_new, v_new)
        for call in range(2):
            qc = q if call == 0 else (q.float() * -0.5).to(torch.bfloat16)
            ref_o = torch.empty((w.B, w.H_Q, w.d_h), device="cuda")
            ref_l = torch.empty((w.B, w.H_Q), device="cuda")
            kvc.kvc_decode_attn(g.pool, 0, qc, g.bt_dec, g.lens_post, ref_o, ref_l, scale=w.scale)
            out = torch.full((w.B, w.H_Q, w.d_h), float("nan"), device="cuda")
            lse = torch.full((w.B, w.H_Q), float("nan"), device="cuda")
            kvc.kvc_decode_attn_noalloc(g.pool, 0, qc, g.bt_dec, g.lens_post, out, lse, scale=w.scale)
            torch.cuda.synchronize()
            assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
            _close(out, lse, ref_o, ref_l, dtype)
    finally:
        g.close()


def test_noalloc_rejects_partials_beyond_the_scratch(kvc):
    """A split plan whose partials exceed 8 MiB is refused before any launch."""
    w = synth.make_workload("custom", B=2, H_Q=32, H_KV=8, d_h=128, lens=[40, 40], extra_cols=2048, seed=4)
    g = GpuCase(kvc, w)
    os.environ["KVC_SPLIT_CHUNK"] = "4"      # 4-block splits over a 2 051-entry table row: 513 splits
    try:
        ld = layer_data(w, 0)
        g.load_context(0, ld)
        q, _, _ = g.step_inputs(ld)
        splits = -(-w.max_blocks // 4)
        assert w.B * w.H_Q * splits * (w.d_h + 2) > SCRATCH_FLOATS
        out = torch.empty((w.B, w.H_Q, w.d_h), device="cuda")
        n0 = kvc.kvc_launch_count()
        with pytest.raises(kvc.KvcError) as e:
            kvc.kvc_decode_attn_noalloc(g.pool, 0, q, g.bt_dec, g.lens_post, out, scale=w.scale)
        assert e.value.status == kvc.KVC_ERR_ARG
        assert kvc.kvc_launch_count() == n0
    finally:
        os.environ.pop("KVC_SPLIT_CHUNK", None)
        g.close()
