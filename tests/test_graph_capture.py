"""A decode step captured in a CUDA graph and replayed gives the eager step's
results bit for bit: with the split merge in the attention kernel (a GQA
layer), as a second, programmatically dependent launch (32-head groups), and
through the allocation-free entry point.  A graph replays the same kernels on
the same inputs, so nothing may differ; what could break is the capture itself
(an allocation, a synchronising call, or the dependent launch's attribute).
"""
import os

import numpy as np
import pytest
import torch

import synth
from harness import GpuCase, layer_data

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", ["gqa_in_kernel_merge", "mqa_merge_launch", "mqa_noalloc"])
def test_graph_replay_equals_eager(kvc, case):
    H_KV = 8 if case == "gqa_in_kernel_merge" else 1
    w = synth.make_workload("custom", B=3, H_Q=32, H_KV=H_KV, d_h=128, lens=[6000, 2500, 40], seed=31)
    # 64-block splits: 6 for the longest sequence, i.e. 4 x 6 partial rows for a group of 4 heads
    # (merged by the last split CTA) and 32 x 6 for 32 heads (merge_kernel)
    os.environ["KVC_SPLIT_CHUNK"] = "64"
    g = GpuCase(kvc, w, fill_byte=0)
    try:
        ld = layer_data(w, 0)
        g.load_context(0, ld)
        q, k_new, v_new = g.step_inputs(ld)

        def call(out, lse):
            if case == "mqa_noalloc":
                kvc.kvc_decode_attn_noalloc(g.pool, 0, q, g.bt_dec, g.lens_post, out, lse, scale=w.scale)
            else:   # the fused step: appending the same rows again stores the same bytes
                kvc.kvc_decode_step(g.pool, 0, q, g.bt_dec, g.lens_pre, k_new, v_new, out, lse, scale=w.scale)

        if case == "mqa_noalloc":
            kvc.kvc_append(g.pool, 0, g.bt_dec, g.lens_pre, k_new, v_new)
        eager_o = torch.empty((w.B, w.H_Q, w.d_h), device="cuda")
        eager_l = torch.empty((w.B, w.H_Q), device="cuda")
        call(eager_o, eager_l)   # first call: kernel set-up and the workspace, outside the capture
        torch.cuda.synchronize()
        before = g.layer_bytes(0)

        out = torch.full_like(eager_o, float("nan"))
        lse = torch.full_like(eager_l, float("nan"))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):   # the binding launches on the capture stream (torch's current one)
            call(out, lse)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
        assert torch.equal(out, eager_o) and torch.equal(lse, eager_l)
        assert np.array_equal(g.layer_bytes(0), before)
    finally:
        g.close()
        os.environ.pop("KVC_SPLIT_CHUNK", None)
