"""kvc_decode_attn_noalloc: decode attention for callers that may not allocate
device memory during a decode step (memory pre-reserved by their own caching
allocator, or loops that cannot afford cudaMalloc's device synchronisation).

It must allocate nothing, give the results of kvc_decode_attn call after call
(its split partials live in the library's fixed per-device scratch array
instead of the pool's workspace), agree with the oracle, and refuse a split
batch whose partials would not fit that array.  Collected last so that a run
stopping at its first failure has run every other test.
"""
import os

import numpy as np
import pytest
import torch

import synth
from harness import GpuCase, OracleCase, check_attention, layer_data

pytestmark = pytest.mark.gpu

SCRATCH_FLOATS = 2 << 20     # the array's documented size: 8 MiB

# (dtype, H_KV, d_h, lens): GQA / MHA / MQA groups, bf16 / e4m3 / int4, both head widths,
# split batches and one short batch that runs unsplit
CASES = [("bf16", 8, 128, [5000, 3000, 17]), ("bf16", 8, 128, [700]), ("bf16", 1, 128, [4000, 33]),
         ("bf16", 32, 128, [2500, 100]), ("bf16", 8, 64, [3000, 9]), ("bf16", 8, 128, [40, 3]),
         ("fp8", 8, 128, [5000, 3000, 17]), ("fp8", 1, 128, [2000, 600]), ("fp8", 32, 128, [1800, 5]),
         ("int4", 8, 128, [4100, 250]), ("int4", 1, 128, [3000, 64])]


@pytest.mark.parametrize("dtype,H_KV,d_h,lens", CASES,
                         ids=[f"{c[0]}-hkv{c[1]}-d{c[2]}-{'x'.join(map(str, c[3]))}" for c in CASES])
def test_noalloc_allocates_nothing_and_matches(kvc, dtype, H_KV, d_h, lens):
    """On a fresh pool (its workspace never sized by kvc_decode_attn): one warm-up
    call, then two calls in a row (the second with new queries, so stale scratch
    cannot pass for a result) with the device's free memory unchanged and one or
    two launches per call; each against the oracle, then against
    kvc_decode_attn (same kernels, partials elsewhere: rounding-level agreement)."""
    w = synth.make_workload("custom", B=len(lens), H_Q=32, H_KV=H_KV, d_h=d_h, lens=lens, dtype=dtype, seed=3)
    g = GpuCase(kvc, w)
    try:
        ld = layer_data(w, 0)
        g.load_context(0, ld)
        q, k_new, v_new = g.step_inputs(ld)
        kvc.kvc_append(g.pool, 0, g.bt_dec, g.lens_pre, k_new, v_new)
        qs = [q, (q.float() * -0.5).to(torch.bfloat16)]
        outs = [torch.full((w.B, w.H_Q, w.d_h), float("nan"), device="cuda") for _ in qs]
        lses = [torch.full((w.B, w.H_Q), float("nan"), device="cuda") for _ in qs]
        ref_o = torch.empty((w.B, w.H_Q, w.d_h), device="cuda")
        ref_l = torch.empty((w.B, w.H_Q), device="cuda")
        kvc.kvc_decode_attn_noalloc(g.pool, 0, qs[0], g.bt_dec, g.lens_post, outs[0], lses[0], scale=w.scale)
        torch.cuda.synchronize()
        free0 = torch.cuda.mem_get_info()[0]
        n0 = kvc.kvc_launch_count()
        for i in range(2):
            kvc.kvc_decode_attn_noalloc(g.pool, 0, qs[i], g.bt_dec, g.lens_post, outs[i], lses[i], scale=w.scale)
        torch.cuda.synchronize()
        launches = kvc.kvc_launch_count() - n0
        assert torch.cuda.mem_get_info()[0] == free0, "device memory changed across allocation-free calls"
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
        assert launches in (2, 4), launches       # attention (+ the split merge) per call

        orc = OracleCase(w).run_layer(ld, image=False)
        check_attention(outs[0], lses[0], orc["out"], orc["lse"], dtype, "noalloc vs oracle")
        for i in range(2):
            kvc.kvc_decode_attn(g.pool, 0, qs[i], g.bt_dec, g.lens_post, ref_o, ref_l, scale=w.scale)
            torch.cuda.synchronize()
            assert torch.equal(torch.isfinite(lses[i]), torch.isfinite(ref_l))
            fin = torch.isfinite(ref_l)
            assert float((outs[i] - ref_o).abs().max()) <= 1e-5
            assert float((lses[i][fin] - ref_l[fin]).abs().max()) <= 1e-5
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
