"""CUDA path vs the oracle, element by element, through the C ABI.

Append and token writes: bit-exact on every byte of the pool (untouched bytes
keep their fill).  Attention: max |out - ref| <= 1e-2 (bf16 KV) / 3e-2 (e4m3
KV) and |lse - ref| <= 2e-3 * max(1, |ref|).  Invariants that the GPU's
arithmetic order cannot change (block permutation, poisoned padding) are
checked bit for bit.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from harness import (GpuCase, OracleCase, check_attention, dev_bits, dev_i32, first_mismatch, layer_data,
                     logical_lists)

pytestmark = pytest.mark.gpu


def _run(kvc, w, layers=(0,), fill=0xFF, bytes_check=True, decode_layers=None, fused=False):
    """Load context, append, decode on the GPU and in the oracle; compare.
    fused: the step as one kvc_decode_step launch (the call bench.py times),
    else kvc_append followed by kvc_decode_attn."""
    g = GpuCase(kvc, w, fill_byte=fill)
    orc = OracleCase(w, fill_byte=fill)
    errs = []
    try:
        for layer in layers:
            ld = layer_data(w, layer)
            g.load_context(layer, ld)
            if fused:
                q, k_new, v_new = g.step_inputs(ld)
                out = torch.empty((w.B, w.H_Q, w.d_h), dtype=torch.float32, device="cuda")
                lse = torch.empty((w.B, w.H_Q), dtype=torch.float32, device="cuda")
                kvc.kvc_decode_step(g.pool, layer, q, g.bt_dec, g.lens_pre, k_new, v_new, out, lse, scale=w.scale)
            else:
                out, lse = g.step(layer, ld)
            torch.cuda.synchronize()
            assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
            dec = decode_layers is None or layer in decode_layers
            ref = orc.run_layer(ld, decode=dec, image=bytes_check)
            if w.dtype != "bf16":
                got_sc = g.pool.scales_view()[layer].cpu().numpy()
                assert np.array_equal(got_sc.view(np.uint32), ref["scales"].view(np.uint32)), "scales differ"
            if bytes_check:
                n, first = first_mismatch(g.layer_bytes(layer), ref["image"].bytes)
                assert n == 0, f"layer {layer}: {n} pool bytes differ, first at {first}"
            if dec:
                errs.append(check_attention(out, lse, ref["out"], ref["lse"], w.dtype, f"{w.name} layer {layer}"))
    finally:
        g.close()
    return errs


# ------------------------------------------------------------------ the workloads
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny(kvc, seed):
    _run(kvc, synth.make_workload("tiny", seed=seed))


@pytest.mark.parametrize("fused", [True, False], ids=["fused_step", "append_then_attend"])
def test_llama_gqa(kvc, fused):
    _run(kvc, synth.make_workload("llama_gqa", seed=0), fused=fused)


@pytest.mark.parametrize("name", ["sweep_hkv8_bf16", "sweep_hkv8_fp8", "sweep_hkv32_bf16", "sweep_hkv32_fp8",
                                  "sweep_hkv1_bf16", "sweep_hkv1_fp8", "sweep_hkv8_int4", "sweep_hkv1_int4",
                                  "sweep_hkv32_int4"])
def test_sweep(kvc, name):
    """Full-size sweep workloads through the fused step, the call bench.py times."""
    _run(kvc, synth.make_workload(name, seed=0), fused=True)


def test_full_pool_graph_replay(kvc):
    """The 32-layer step of the 32 GiB pool exactly as bench.py times it: one
    eager step (kernel set-up, workspace), then the 32 fused kvc_decode_step
    launches captured in one CUDA graph and replayed into NaN-filled outputs.
    Every layer's pool bytes bit-exact against the oracle's image; attention of
    four layers (first, last and two inside) against the oracle.  Appending the
    same rows at the same positions again stores the same bytes, so the eager
    step and the replay leave one state."""
    w = synth.make_workload("full_pool", seed=0)
    g = GpuCase(kvc, w, fill_byte=0xFF)
    try:
        ins, outs = [], []
        for layer in range(w.L):
            ld = layer_data(w, layer)
            g.load_context(layer, ld)
            ins.append(g.step_inputs(ld))
            outs.append((torch.empty((w.B, w.H_Q, w.d_h), device="cuda"), torch.empty((w.B, w.H_Q), device="cuda")))
            del ld
        torch.cuda.synchronize()

        def step():
            for layer in range(w.L):
                q, k_new, v_new = ins[layer]
                kvc.kvc_decode_step(g.pool, layer, q, g.bt_dec, g.lens_pre, k_new, v_new, *outs[layer], scale=w.scale)

        step()
        torch.cuda.synchronize()
        for o, l in outs:
            o.fill_(float("nan"))
            l.fill_(float("nan"))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        graph.replay()
        torch.cuda.synchronize()
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
        orc = OracleCase(w, fill_byte=0xFF)
        for layer in range(w.L):
            ld = layer_data(w, layer)
            dec = layer in (0, 7, 20, 31)
            ref = orc.run_layer(ld, decode=dec)
            n, first = first_mismatch(g.layer_bytes(layer), ref["image"].bytes)
            assert n == 0, f"layer {layer}: {n} pool bytes differ, first at {first}"
            if dec:
                check_attention(outs[layer][0], outs[layer][1], ref["out"], ref["lse"], "bf16", f"full pool layer {layer}")
            del ld, ref
    finally:
        g.close()


def test_ragged_prefix_and_prefill_chunk(kvc):
    w = synth.make_workload("ragged_prefix", seed=0)
    g = GpuCase(kvc, w)
    orc = OracleCase(w)
    try:
        ld = layer_data(w, 0)
        g.load_context(0, ld)
        out, lse = g.step(0, ld)
        ref = orc.run_layer(ld)
        check_attention(out, lse, ref["out"], ref["lse"], "bf16", "ragged decode")
        # the 600-token chunk of row 64: written after the shared 1200-token prefix, then causal attention
        p = w.prefill
        kc = w.ctx_tokens(0, 0, p.seq, p.q_start, p.total)
        vc = w.ctx_tokens(0, 1, p.seq, p.q_start, p.total)
        row = dev_i32(w.block_tables[p.seq:p.seq + 1])
        kvc.kvc_write_tokens(g.pool, 0, row, dev_i32([p.q_start]), dev_i32([0, p.n_q]), dev_bits(kc), dev_bits(vc))
        qc = w.prefill_q(0)
        o2 = torch.empty((p.n_q, w.H_Q, w.d_h), dtype=torch.float32, device="cuda")
        l2 = torch.empty((p.n_q, w.H_Q), dtype=torch.float32, device="cuda")
        kvc.kvc_prefill_attn(g.pool, 0, dev_bits(qc), row[0], p.q_start, o2, l2, scale=w.scale)
        torch.cuda.synchronize()
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
        shared_k, shared_v = ld.k_ctx[:w.shared_prefix], ld.v_ctx[:w.shared_prefix]
        K = np.concatenate([shared_k, kc])
        V = np.concatenate([shared_v, vc])
        ro, rl = oracle.prefill(qc, K, V, p.q_start, w.H_KV, scale=w.scale)
        check_attention(o2, l2, ro, rl, "bf16", "prefill chunk")
        # pool bytes, prefill chunk included
        ref["image"].write_tokens(0, w.block_tables[p.seq:p.seq + 1], np.array([p.q_start], np.int32),
                                  np.array([0, p.n_q], np.int64), kc, vc)
        n, first = first_mismatch(g.layer_bytes(0), ref["image"].bytes)
        assert n == 0, f"{n} pool bytes differ, first at {first}"
    finally:
        g.close()


@pytest.mark.parametrize("case", ["ragged_prefix", "small", "fp8", "int4", "mqa"])
def test_mixed_step_equals_step_then_prefill(kvc, case):
    """kvc_mixed_step (a decode step and a prefill chunk together) leaves the
    pool bytes of kvc_decode_step followed by kvc_prefill_attn and gives their
    outputs: bit-identical for bf16 pools (the same kernels and split plans),
    and decode and prefill both within tolerance of the oracle.  e4m3 and int4
    pools run it as one launch of the mixed kernel (fewer launches than the two
    calls); bf16 pools run the decode launch with the tensor-memory prefill
    kernel as its programmatic dependent (the same launches as the two calls)."""
    kw = {"ragged_prefix": {},
          "small": dict(B=6, shared=96, chunk=70, lo=16, hi=900),
          "fp8": dict(B=6, shared=96, chunk=70, lo=16, hi=900, dtype="fp8"),
          "int4": dict(B=6, shared=96, chunk=70, lo=16, hi=900, dtype="int4"),
          "mqa": dict(B=3, shared=48, chunk=33, lo=16, hi=300, H_KV=1)}[case]
    w = synth.make_workload("ragged_prefix", seed=1, **kw)
    p = w.prefill
    ld = layer_data(w, 0)
    kc = w.ctx_tokens(0, 0, p.seq, p.q_start, p.total)
    vc = w.ctx_tokens(0, 1, p.seq, p.q_start, p.total)
    qc = w.prefill_q(0)
    res = []
    for mixed in (False, True):
        g = GpuCase(kvc, w, fill_byte=0xA5)
        try:
            g.load_context(0, ld)
            row = dev_i32(w.block_tables[p.seq:p.seq + 1])
            kvc.kvc_write_tokens(g.pool, 0, row, dev_i32([p.q_start]), dev_i32([0, p.n_q]), dev_bits(kc), dev_bits(vc))
            q, k, v = g.step_inputs(ld)
            out = torch.empty((w.B, w.H_Q, w.d_h), device="cuda")
            lse = torch.empty((w.B, w.H_Q), device="cuda")
            o2 = torch.empty((p.n_q, w.H_Q, w.d_h), device="cuda")
            l2 = torch.empty((p.n_q, w.H_Q), device="cuda")
            n0 = kvc.kvc_launch_count()
            if mixed:
                kvc.kvc_mixed_step(g.pool, 0, q, g.bt_dec, g.lens_pre, k, v, out, lse, dev_bits(qc), row[0],
                                   p.q_start, o2, l2, scale=w.scale)
            else:
                kvc.kvc_decode_step(g.pool, 0, q, g.bt_dec, g.lens_pre, k, v, out, lse, scale=w.scale)
                kvc.kvc_prefill_attn(g.pool, 0, dev_bits(qc), row[0], p.q_start, o2, l2, scale=w.scale)
            torch.cuda.synchronize()
            assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
            res.append((g.layer_bytes(0), out.cpu(), lse.cpu(), o2.cpu(), l2.cpu(), kvc.kvc_launch_count() - n0))
        finally:
            g.close()
    n, first = first_mismatch(res[0][0], res[1][0])
    assert n == 0, f"{n} pool bytes differ, first at {first}"
    if w.dtype != "bf16":
        assert res[1][5] < res[0][5], "the mixed kernel should take fewer launches"
    else:
        assert res[1][5] == res[0][5]
    if w.dtype == "bf16":
        for a, b in zip(res[0][1:5], res[1][1:5]):
            assert torch.equal(a, b)
    ref = OracleCase(w).run_layer(ld, image=False)
    check_attention(res[1][1], res[1][2], ref["out"], ref["lse"], w.dtype, f"mixed decode {case}")
    sc = ref["scales"]
    K = np.concatenate([ld.k_ctx[:w.shared_prefix], kc])
    V = np.concatenate([ld.v_ctx[:w.shared_prefix], vc])
    if sc is not None:
        qz = oracle.quantize_e4m3 if w.dtype == "fp8" else oracle.quantize_int4
        K, V = qz(K, sc[0]), qz(V, sc[1])
    ro, rl = oracle.prefill(qc, K, V, p.q_start, w.H_KV, scales=sc, scale=w.scale, kind=w.dtype)
    check_attention(res[1][3], res[1][4], ro, rl, w.dtype, f"mixed prefill {case}")


def test_mixed_step_edges(kvc):
    """kvc_mixed_step with no chunk queries is kvc_decode_step, with no decode
    sequences is kvc_prefill_attn (bit-identical outputs); a chunk running past its
    row or a misaligned q is refused before any launch."""
    w = synth.make_workload("ragged_prefix", seed=3, B=3, shared=32, chunk=21, lo=16, hi=300)
    p = w.prefill
    ld = layer_data(w, 0)
    kc = w.ctx_tokens(0, 0, p.seq, p.q_start, p.total)
    vc = w.ctx_tokens(0, 1, p.seq, p.q_start, p.total)
    qc = dev_bits(w.prefill_q(0))
    g = GpuCase(kvc, w)
    try:
        g.load_context(0, ld)
        row = dev_i32(w.block_tables[p.seq])
        kvc.kvc_write_tokens(g.pool, 0, row[None], dev_i32([p.q_start]), dev_i32([0, p.n_q]), dev_bits(kc), dev_bits(vc))
        q, k, v = g.step_inputs(ld)
        outs = [torch.empty((w.B, w.H_Q, w.d_h), device="cuda") for _ in range(2)]
        lses = [torch.empty((w.B, w.H_Q), device="cuda") for _ in range(2)]
        o2 = [torch.empty((p.n_q, w.H_Q, w.d_h), device="cuda") for _ in range(2)]
        l2 = [torch.empty((p.n_q, w.H_Q), device="cuda") for _ in range(2)]
        # no chunk queries: the decode step alone (same append position, so the pool is unchanged)
        kvc.kvc_decode_step(g.pool, 0, q, g.bt_dec, g.lens_pre, k, v, outs[0], lses[0], scale=w.scale)
        kvc.kvc_mixed_step(g.pool, 0, q, g.bt_dec, g.lens_pre, k, v, outs[1], lses[1], qc[:0], row, p.q_start,
                           o2[1][:0], l2[1][:0], scale=w.scale)
        # no decode sequences: the chunk alone
        kvc.kvc_prefill_attn(g.pool, 0, qc, row, p.q_start, o2[0], l2[0], scale=w.scale)
        kvc.kvc_mixed_step(g.pool, 0, q[:0], g.bt_dec[:0], g.lens_pre[:0], k[:0], v[:0], outs[1][:0], lses[1][:0],
                           qc, row, p.q_start, o2[1], l2[1], scale=w.scale)
        torch.cuda.synchronize()
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
        assert torch.equal(outs[0], outs[1]) and torch.equal(lses[0], lses[1])
        assert torch.equal(o2[0], o2[1]) and torch.equal(l2[0], l2[1])
        with pytest.raises(kvc.KvcError) as e:    # the chunk's last query would sit past the row's table
            kvc.kvc_mixed_step(g.pool, 0, q, g.bt_dec, g.lens_pre, k, v, outs[1], lses[1], qc, row,
                               w.max_blocks * 16 - p.n_q + 1, o2[1], l2[1], scale=w.scale)
        assert e.value.status == kvc.KVC_ERR_RANGE
        qbad = torch.empty(q.numel() * 2 + 8, dtype=torch.bfloat16, device="cuda")[1:1 + q.numel()].view(q.shape)
        with pytest.raises(kvc.KvcError) as e:    # q not 16-byte aligned
            kvc.kvc_mixed_step(g.pool, 0, qbad, g.bt_dec, g.lens_pre, k, v, outs[1], lses[1], qc, row, p.q_start,
                               o2[1], l2[1], scale=w.scale)
        assert e.value.status == kvc.KVC_ERR_ARG
        torch.cuda.synchronize()
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
    finally:
        g.close()


def test_prefix_sharing_equals_private_copies(kvc):
    """The shared-block run equals a run where every row holds a private copy
    of the prefix blocks: bit-identical outputs (same arithmetic order)."""
    w = synth.make_workload("ragged_prefix", seed=1)
    g = GpuCase(kvc, w)
    try:
        ld = layer_data(w, 0)
        g.load_context(0, ld)
        out_a, lse_a = [t.clone() for t in g.step(0, ld)]
    finally:
        g.close()
    # private copies: remap each row's prefix blocks to fresh ids appended to the pool
    sb = w.shared_prefix // w.bs
    bt = w.block_tables.copy()
    N0 = w.num_blocks
    for r in range(w.B):
        bt[r, :sb] = N0 + r * sb + np.arange(sb, dtype=np.int32)
    w2 = synth.workloads.Workload(w.name, w.seed, w.B, w.H_Q, w.H_KV, w.d_h, w.bs, w.L, w.dtype,
                                  N0 + w.B * sb, w.lens_pre, bt[:w.B])
    ld2 = layer_data(w2, 0)
    # same values: the rows' prefixes come from the shared stream in w; copy them in as private context
    ks, vs, cu = [], [], [0]
    for b in range(w.B):
        a, e = int(ld.cu[1 + b]), int(ld.cu[2 + b])
        ks += [ld.k_ctx[:w.shared_prefix], ld.k_ctx[a:e]]
        vs += [ld.v_ctx[:w.shared_prefix], ld.v_ctx[a:e]]
        cu.append(cu[-1] + w.shared_prefix + e - a)
    ld2.k_ctx, ld2.v_ctx = np.concatenate(ks), np.concatenate(vs)
    ld2.cu, ld2.start, ld2.rows = np.array(cu, np.int32), np.zeros(w.B, np.int32), np.arange(w.B, dtype=np.int32)
    ld2.q, ld2.k_new, ld2.v_new = ld.q, ld.k_new, ld.v_new
    g2 = GpuCase(kvc, w2)
    try:
        g2.load_context(0, ld2)
        out_b, lse_b = g2.step(0, ld2)
        assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)
    finally:
        g2.close()


# ------------------------------------------------------------------ edge cases
def _custom(**kw):
    return synth.make_workload("custom", **kw)


@pytest.mark.parametrize("d_h", [64, 128])
def test_short_and_boundary_lengths(kvc, d_h):
    """First token (empty context), lengths on and around block boundaries, a
    ragged tail in the last block, over several split sizes."""
    lens = [0, 1, 14, 15, 16, 17, 31, 32, 33, 47, 64, 100, 255, 511]
    w = _custom(B=len(lens), H_Q=8, H_KV=2, d_h=d_h, lens=lens, spare_blocks=5, extra_cols=3)
    for chunk in (None, "4", "8", "16"):
        if chunk:
            os.environ["KVC_SPLIT_CHUNK"] = chunk
        try:
            _run(kvc, w)
        finally:
            os.environ.pop("KVC_SPLIT_CHUNK", None)


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "int4"])
@pytest.mark.parametrize("H_KV", [32, 16, 8, 4, 2, 1])
def test_group_sizes(kvc, H_KV, dtype):
    """GQA group sizes 1 (MHA) .. 32 (MQA) with ragged lengths."""
    lens = [3, 77, 300, 1029]
    _run(kvc, _custom(B=len(lens), H_Q=32, H_KV=H_KV, d_h=128, lens=lens, dtype=dtype, seed=H_KV))


def _f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)   # round to nearest even (finite x)


@pytest.mark.parametrize("dtype", ["bf16", "fp8", "int4"])
@pytest.mark.parametrize("H_KV", [8, 1])
def test_rising_and_falling_scores(kvc, dtype, H_KV):
    """Scores that climb along a sequence by about 2 (log2 units) per block, so a
    running maximum is overtaken within the rescale slack for several blocks and
    then past it; one sequence whose scores fall (its maximum stays in the first
    block); one random sequence.  Every query leans on one direction u (q = n + 1,
    k_t = n_t + a(t)), so q.k_t grows with a(t) for every head."""
    lens = [700, 1500, 333, 2048]
    w = _custom(B=len(lens), H_Q=32, H_KV=H_KV, d_h=128, lens=lens, dtype=dtype, seed=11 + H_KV)
    ld = layer_data(w, 0)
    slope = 0.12 / 16    # a(t) per position: ~2 log2 units of score per 16-position block
    ramp = {0: slope, 1: slope, 2: -slope, 3: 0.0}
    k = synth.bf16_bits_to_f32(ld.k_ctx).astype(np.float32)
    for i in range(len(ld.rows)):
        b, t0, n = int(ld.rows[i]), int(ld.start[i]), int(ld.cu[i + 1] - ld.cu[i])
        t = np.arange(t0, t0 + n, dtype=np.float32)
        a = ramp[b] * (t if ramp[b] >= 0 else t - t0 - n)
        k[ld.cu[i]:ld.cu[i + 1]] += a[:, None, None]
    ld.k_ctx = _f32_to_bf16_bits(k)
    kn = synth.bf16_bits_to_f32(ld.k_new).astype(np.float32)
    kn += np.array([ramp[b] * lens[b] if ramp[b] >= 0 else 0.0 for b in range(w.B)], np.float32)[:, None, None]
    ld.k_new = _f32_to_bf16_bits(kn)
    ld.q = _f32_to_bf16_bits(synth.bf16_bits_to_f32(ld.q).astype(np.float32) + 1.0)
    for chunk in (None, "8", "40"):
        if chunk:
            os.environ["KVC_SPLIT_CHUNK"] = chunk
        g = GpuCase(kvc, w, fill_byte=0xFF)
        try:
            g.load_context(0, ld)
            out, lse = g.step(0, ld)
            torch.cuda.synchronize()
            assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
        finally:
            g.close()
            os.environ.pop("KVC_SPLIT_CHUNK", None)
        ref = OracleCase(w, fill_byte=0xFF).run_layer(ld, image=False)
        check_attention(out, lse, ref["out"], ref["lse"], w.dtype, f"rising scores {dtype} H_KV={H_KV} chunk={chunk}")
        # the scores really climb: the newest position's lse is tens of log2 units above a random one's
        assert float(ref["lse"][0].min()) > float(ref["lse"][3].max()) + 20


@pytest.mark.parametrize("case", ["in_kernel_65_splits", "in_kernel_32_heads", "merge_kernel_1032_splits"])
def test_merge_paths(kvc, case):
    """The split merge past its fast paths, against the oracle: the last split CTA
    merging more than 32 splits (its lanes loop) or 32 query heads' rows, and
    merge_kernel over more splits than it keeps weights for in shared memory
    (1 024; the rest are recomputed) and than a thread preloads."""
    env = {"in_kernel_65_splits": dict(KVC_SPLIT_CHUNK="4", KVC_MERGE_ROWS="4096"),
           "in_kernel_32_heads": dict(KVC_SPLIT_CHUNK="16", KVC_MERGE_ROWS="4096"),
           "merge_kernel_1032_splits": dict(KVC_SPLIT_CHUNK="4")}[case]
    shape = {"in_kernel_65_splits": dict(H_Q=8, H_KV=8, lens=[4096, 1000]),
             "in_kernel_32_heads": dict(H_Q=32, H_KV=1, lens=[4096, 77]),
             "merge_kernel_1032_splits": dict(H_Q=4, H_KV=1, lens=[65999, 3])}[case]
    w = _custom(B=len(shape["lens"]), H_Q=shape["H_Q"], H_KV=shape["H_KV"], d_h=128, lens=shape["lens"], seed=23)
    os.environ.update(env)
    try:
        _run(kvc, w, bytes_check=False)
    finally:
        for k in env:
            os.environ.pop(k, None)


def test_split_counts_agree(kvc):
    """Changing the split size changes only rounding: all within tolerance of the oracle."""
    w = _custom(B=3, H_Q=16, H_KV=4, d_h=128, lens=[2000, 4097, 777])
    for chunk in ("4", "12", "64", "1024"):
        os.environ["KVC_SPLIT_CHUNK"] = chunk
        try:
            _run(kvc, w, bytes_check=False)
        finally:
            os.environ.pop("KVC_SPLIT_CHUNK", None)


@pytest.mark.parametrize("case", ["many_splits", "many_short", "large_batch", "fp8", "int4"])
def test_batch_shapes(kvc, case):
    """Batches whose split plans differ: long sequences over many splits merged
    by their last CTA, many short sequences (first tokens included), a batch of
    1 025 sequences, e4m3 and int4 pools with lengths from 1 to 5 001."""
    rng = np.random.default_rng(7)
    w = {"many_splits": lambda: _custom(B=8, H_Q=16, H_KV=4, d_h=128, lens=[3000, 2999, 3001, 2048, 1, 9000, 17, 3333]),
         "many_short": lambda: _custom(B=300, H_Q=8, H_KV=1, d_h=64, lens=rng.integers(0, 41, 300), seed=3),
         "large_batch": lambda: _custom(B=1025, H_Q=8, H_KV=1, d_h=128, lens=rng.integers(0, 70, 1025), seed=5),
         "fp8": lambda: _custom(B=6, H_Q=32, H_KV=8, d_h=128, lens=[5000, 1, 0, 2500, 777, 4096], dtype="fp8"),
         "int4": lambda: _custom(B=6, H_Q=32, H_KV=8, d_h=128, lens=[5000, 1, 0, 2500, 777, 4096], dtype="int4")}[case]()
    _run(kvc, w, bytes_check=case != "large_batch")


def test_block_permutation_bit_identical(kvc):
    """Same logical sequences, physical blocks permuted and tables rewritten:
    bit-identical outputs (logical order is what attention sees)."""
    w = _custom(B=4, H_Q=32, H_KV=8, d_h=128, lens=[700, 1300, 64, 2049], spare_blocks=11)
    res = []
    for perm_seed in (0, 1):
        remap = synth.permutation(perm_seed, 77, w.num_blocks)
        bt = np.where(w.block_tables >= 0, remap[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
        w2 = synth.workloads.Workload(w.name, w.seed, w.B, w.H_Q, w.H_KV, w.d_h, w.bs, w.L, w.dtype,
                                      w.num_blocks, w.lens_pre, bt)
        g = GpuCase(kvc, w2)
        try:
            ld = layer_data(w2, 0)
            g.load_context(0, ld)
            res.append([t.clone() for t in g.step(0, ld)])
        finally:
            g.close()
    assert torch.equal(res[0][0], res[1][0]) and torch.equal(res[0][1], res[1][1])


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_padding_poison_bit_identical(kvc, dtype):
    """Pool pre-filled with NaN/Inf patterns vs zeros: unused slots and blocks
    never change the output ("KV cache: ..." 21.1: padded slots are excluded)."""
    w = _custom(B=5, H_Q=32, H_KV=8, d_h=128, lens=[1, 17, 250, 1000, 33], spare_blocks=9, dtype=dtype)
    res = []
    for fill in (0x00, 0xFF, 0x7F):
        g = GpuCase(kvc, w, fill_byte=fill)
        try:
            ld = layer_data(w, 0)
            g.load_context(0, ld)
            res.append([t.clone() for t in g.step(0, ld)])
        finally:
            g.close()
    for r in res[1:]:
        assert torch.equal(res[0][0], r[0]) and torch.equal(res[0][1], r[1])


def test_head_duplication_agrees(kvc):
    """MQA data duplicated into 8 and 32 KV heads gives the same attention (within tolerance)."""
    lens = [130, 900]
    w1 = _custom(B=2, H_Q=32, H_KV=1, d_h=128, lens=lens)
    ld1 = layer_data(w1, 0)
    outs = []
    for H_KV in (1, 8, 32):
        w = _custom(B=2, H_Q=32, H_KV=H_KV, d_h=128, lens=lens)
        ld = layer_data(w, 0)
        ld.k_ctx, ld.v_ctx = np.repeat(ld1.k_ctx, H_KV, 1), np.repeat(ld1.v_ctx, H_KV, 1)
        ld.k_new, ld.v_new, ld.q = np.repeat(ld1.k_new, H_KV, 1), np.repeat(ld1.v_new, H_KV, 1), ld1.q
        g = GpuCase(kvc, w)
        try:
            g.load_context(0, ld)
            outs.append([t.cpu().numpy() for t in g.step(0, ld)])
        finally:
            g.close()
    ref = OracleCase(w1).run_layer(ld1, image=False)
    for o, l in outs:
        check_attention(o, l, ref["out"], ref["lse"], "bf16", "duplicated heads")


def test_empty_batch_and_empty_sequence(kvc):
    w = _custom(B=2, H_Q=8, H_KV=2, d_h=128, lens=[5, 9])
    g = GpuCase(kvc, w)
    try:
        q = torch.zeros((0, 8, 128), dtype=torch.bfloat16, device="cuda")
        out = torch.empty((0, 8, 128), dtype=torch.float32, device="cuda")
        kvc.kvc_decode_attn(g.pool, 0, q, g.bt_dec[:0], g.lens_post[:0], out)   # B = 0: no-op
        ld = layer_data(w, 0)
        g.load_context(0, ld)
        q, _, _ = g.step_inputs(ld)
        out = torch.full((2, 8, 128), 7.0, device="cuda")
        lse = torch.full((2, 8), 7.0, device="cuda")
        kvc.kvc_decode_attn(g.pool, 0, q, g.bt_dec, dev_i32([0, 3]), out, lse, scale=w.scale)
        torch.cuda.synchronize()
        assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
        assert torch.all(torch.isfinite(out[1])) and torch.all(torch.isfinite(lse[1]))
        out.fill_(7.0)
        lse.fill_(7.0)
        kvc.kvc_decode_attn(g.pool, 0, q, g.bt_dec, dev_i32([0, 0]), out, lse, scale=w.scale)   # nothing to read
        torch.cuda.synchronize()
        assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
    finally:
        g.close()


def test_device_detected_errors_do_not_fault(kvc):
    """A table entry outside the pool or a length past the table row is
    skipped and reported by kvc_pool_sync_status; the pool stays usable."""
    w = _custom(B=2, H_Q=8, H_KV=2, d_h=128, lens=[40, 20], spare_blocks=2)
    g = GpuCase(kvc, w, fill_byte=0)
    try:
        ld = layer_data(w, 0)
        g.load_context(0, ld)
        before = g.layer_bytes(0)
        bad = w.block_tables.copy()
        bad[0, 40 // 16] = w.num_blocks + 5          # the block the append of row 0 lands in
        q, k, v = g.step_inputs(ld)
        kvc.kvc_append(g.pool, 0, dev_i32(bad), g.lens_pre, k, v)
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_ERR_BAD_BLOCK
        after = g.layer_bytes(0)
        # row 1's append landed, row 0's was skipped
        img = oracle.PoolImage(w.num_blocks, w.bs, 1, w.H_KV, w.d_h, 2)
        img.bytes[:] = before
        img.append(0, bad, w.lens_pre, ld.k_new, ld.v_new)
        assert np.array_equal(after, img.bytes)
        out = torch.empty((2, 8, 128), device="cuda")
        kvc.kvc_decode_attn(g.pool, 0, q, dev_i32(bad), g.lens_post, out, scale=w.scale)
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_ERR_BAD_BLOCK
        too_long = dev_i32([w.max_blocks * 16 + 1, 3])
        kvc.kvc_decode_attn(g.pool, 0, q, g.bt_dec, too_long, out, scale=w.scale)
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_ERR_RANGE
        assert torch.all(out[0] == 0)
        kvc.kvc_decode_attn(g.pool, 0, q, g.bt_dec, g.lens_post, out, scale=w.scale)
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
    finally:
        g.close()


def test_host_argument_errors(kvc):
    w = _custom(B=1, H_Q=8, H_KV=2, d_h=128, lens=[5])
    g = GpuCase(kvc, w)
    try:
        q = torch.zeros((1, 6, 128), dtype=torch.bfloat16, device="cuda")     # 6 % 4 KV heads... H_Q % H_KV != 0
        q7 = torch.zeros((1, 7, 128), dtype=torch.bfloat16, device="cuda")
        out = torch.empty((1, 7, 128), device="cuda")
        with pytest.raises(kvc.KvcError) as e:
            kvc.kvc_decode_attn(g.pool, 0, q7, g.bt_dec, g.lens_post, out)
        assert e.value.status == kvc.KVC_ERR_ARG
        with pytest.raises(kvc.KvcError) as e:
            kvc.kvc_decode_attn(g.pool, 1, q, g.bt_dec, g.lens_post, out)      # layer out of range
        assert e.value.status == kvc.KVC_ERR_ARG
        with pytest.raises(kvc.KvcError) as e:
            kvc.kvc_prefill_attn(g.pool, 0, q, g.bt_dec[0], w.max_blocks * 16, out)
        assert e.value.status == kvc.KVC_ERR_RANGE
    finally:
        g.close()
    with pytest.raises(kvc.KvcError):
        kvc.kvc_pool_create(10, 16, 1, 2, 96, kvc.KVC_BF16)                     # head_dim 96 unsupported


def test_table_21_1_through_the_abi(kvc):
    """Table 21.1 replayed on a real pool with 4-position blocks: A=[7,2] holds 6
    tokens, B=[9] holds 4; A's positions 6, 7 land in block 2 slots 2, 3 and,
    once block 5 is mapped, position 8 in block 5 slot 0; B is untouched."""
    N, bs, H, d = 10, 4, 1, 64
    pool = kvc.kvc_pool_create(N, bs, 1, H, d, kvc.KVC_BF16)
    try:
        pool.bytes_view().fill_(0)
        img = oracle.PoolImage(N, bs, 1, H, d, 2, fill=0)
        bt = np.array([[7, 2, -1], [9, -1, -1]], dtype=np.int32)
        ctx = synth.normal_bf16(5, 1, 10 * H * d).reshape(10, H, d)
        cu = np.array([0, 6, 10], np.int32)
        kvc.kvc_write_tokens(pool, 0, dev_i32(bt), dev_i32([0, 0]), dev_i32(cu), dev_bits(ctx), dev_bits(ctx))
        img.write_tokens(0, bt, np.array([0, 0], np.int32), cu.astype(np.int64), ctx, ctx)
        for pos, extend in ((6, None), (7, None), (8, 5)):
            if extend is not None:
                bt[0, 2] = extend
            k = synth.normal_bf16(6, pos, H * d).reshape(1, H, d)
            kvc.kvc_append(pool, 0, dev_i32(bt[:1]), dev_i32([pos]), dev_bits(k), dev_bits(k))
            img.append(0, bt[:1], np.array([pos], np.int32), k, k)
            torch.cuda.synchronize()
            assert kvc.kvc_pool_sync_status(pool) == kvc.KVC_OK
            assert np.array_equal(pool.bytes_view().cpu().numpy(), img.bytes)
        # where the three appends landed (Table 21.1 steps 1-2)
        got = pool.bytes_view().cpu().numpy()
        for pos, (phys, slot) in ((6, (2, 2)), (7, (2, 3)), (8, (5, 0))):
            k = synth.normal_bf16(6, pos, H * d)
            off = img.offset(0, phys, 0, 0, slot, 0) * 2
            assert np.array_equal(got[off:off + 2 * d].view(np.uint16), k)
    finally:
        pool.close()


@pytest.mark.parametrize("scale", [1.0, 1.0 / 448, 0.0123, 2.0 ** -10])
def test_e4m3_append_matches_codec_for_every_bf16(kvc, scale):
    """Every bf16 bit pattern appended through an e4m3 pool: the stored code is
    the oracle's RNE-saturating encoding of fp32(x) / scale (NaN inputs: NaN codes)."""
    H, d = 1, 128
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    n_tok = 65536 // (H * d)
    N = n_tok // 16
    pool = kvc.kvc_pool_create(N, 16, 1, H, d, kvc.KVC_FP8_E4M3)
    try:
        s = torch.full((H, d), scale, dtype=torch.float32, device="cuda")
        kvc.kvc_pool_set_scales(pool, 0, s, s)
        x = bits.reshape(n_tok, H, d)
        bt = np.arange(N, dtype=np.int32).reshape(1, N)
        kvc.kvc_write_tokens(pool, 0, dev_i32(bt), dev_i32([0]), dev_i32([0, n_tok]), dev_bits(x), dev_bits(x))
        torch.cuda.synchronize()
        img = oracle.PoolImage(N, 16, 1, H, d, 1)
        img.scales[0] = np.float32(scale)
        img.write_tokens(0, bt, np.array([0], np.int32), np.array([0, n_tok], np.int64), x, x)
        got = pool.bytes_view().cpu().numpy()
        xf = synth.bf16_bits_to_f32(bits)
        st, kg, _ = img.gather(0, bt[0], n_tok)
        # locate each input's stored code in both images
        pos_codes_gpu = np.empty(65536, np.uint8)
        gimg = oracle.PoolImage(N, 16, 1, H, d, 1)
        gimg.bytes[:] = got
        _, kgg, _ = gimg.gather(0, bt[0], n_tok)
        pos_codes_gpu[:] = kgg.reshape(-1)
        ref = kg.reshape(-1)
        nan_in = np.isnan(xf)
        assert np.array_equal(pos_codes_gpu[~nan_in], ref[~nan_in])
        assert np.all((pos_codes_gpu[nan_in] & 0x7F) == 0x7F)
    finally:
        pool.close()


def test_launches_are_counted(kvc):
    w = synth.make_workload("tiny", seed=0)
    g = GpuCase(kvc, w)
    try:
        ld = layer_data(w, 0)
        g.load_context(0, ld)
        n0 = kvc.kvc_launch_count()
        g.step(0, ld)
        assert kvc.kvc_launch_count() - n0 >= 2
    finally:
        g.close()


@pytest.mark.parametrize("case", ["tiny", "boundary", "boundary_split4", "fp8_gqa", "mqa", "mha_fp8", "int4_gqa",
                                  "int4_mqa"])
def test_fused_step_equals_append_then_decode(kvc, case):
    """kvc_decode_step (append + attention in one launch) leaves the same pool
    bytes and gives bit-identical outputs to kvc_append then kvc_decode_attn."""
    lens = [0, 1, 15, 16, 31, 100, 1023]
    w = {"tiny": lambda: synth.make_workload("tiny", seed=1),
         "boundary": lambda: _custom(B=len(lens), H_Q=32, H_KV=8, d_h=128, lens=lens),
         "boundary_split4": lambda: _custom(B=len(lens), H_Q=32, H_KV=8, d_h=128, lens=lens),
         "fp8_gqa": lambda: _custom(B=3, H_Q=32, H_KV=8, d_h=128, lens=[7, 500, 2047], dtype="fp8"),
         "mqa": lambda: _custom(B=2, H_Q=32, H_KV=1, d_h=128, lens=[300, 65]),
         "mha_fp8": lambda: _custom(B=2, H_Q=16, H_KV=16, d_h=128, lens=[48, 17], dtype="fp8"),
         "int4_gqa": lambda: _custom(B=3, H_Q=32, H_KV=8, d_h=128, lens=[0, 300, 1025], dtype="int4"),
         "int4_mqa": lambda: _custom(B=2, H_Q=32, H_KV=1, d_h=128, lens=[77, 15], dtype="int4")}[case]()
    if case == "boundary_split4":
        os.environ["KVC_SPLIT_CHUNK"] = "4"
    try:
        ld = layer_data(w, 0)
        res = []
        for fused in (False, True):
            g = GpuCase(kvc, w, fill_byte=0xA5)
            try:
                g.load_context(0, ld)
                q, k, v = g.step_inputs(ld)
                out = torch.empty((w.B, w.H_Q, w.d_h), device="cuda")
                lse = torch.empty((w.B, w.H_Q), device="cuda")
                if fused:
                    kvc.kvc_decode_step(g.pool, 0, q, g.bt_dec, g.lens_pre, k, v, out, lse, scale=w.scale)
                else:
                    kvc.kvc_append(g.pool, 0, g.bt_dec, g.lens_pre, k, v)
                    kvc.kvc_decode_attn(g.pool, 0, q, g.bt_dec, g.lens_post, out, lse, scale=w.scale)
                torch.cuda.synchronize()
                assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
                res.append((g.layer_bytes(0), out.cpu(), lse.cpu()))
            finally:
                g.close()
        n, first = first_mismatch(res[0][0], res[1][0])
        assert n == 0, f"{n} pool bytes differ, first at {first}"
        assert torch.equal(res[0][1], res[1][1]) and torch.equal(res[0][2], res[1][2])
        ref = OracleCase(w).run_layer(ld, image=False)
        check_attention(res[1][1], res[1][2], ref["out"], ref["lse"], w.dtype, f"fused {case}")
    finally:
        os.environ.pop("KVC_SPLIT_CHUNK", None)


def test_copy_blocks_every_layer(kvc):
    """kvc_copy_blocks copies a block's keys and values in every layer, bit for bit."""
    N, L, H, d = 12, 3, 2, 128
    pool = kvc.kvc_pool_create(N, 16, L, H, d, kvc.KVC_BF16)
    try:
        view = pool.bytes_view()
        src = torch.from_numpy(synth.u64(9, 1, view.numel() // 8).view(np.uint8).copy()).cuda()
        view.copy_(src)
        pairs = [(3, 7), (0, 11), (5, 5)]
        kvc.kvc_copy_blocks(pool, dev_i32(np.array(pairs, np.int32)))
        torch.cuda.synchronize()
        assert kvc.kvc_pool_sync_status(pool) == kvc.KVC_OK
        ref = src.cpu().numpy().copy()
        blk = 2 * H * 16 * d * 2
        per_layer = N * blk
        for l in range(L):
            for s, t in pairs:
                ref[l * per_layer + t * blk:l * per_layer + (t + 1) * blk] = \
                    ref[l * per_layer + s * blk:l * per_layer + (s + 1) * blk]
        assert np.array_equal(view.cpu().numpy(), ref)
        kvc.kvc_copy_blocks(pool, dev_i32(np.array([[1, N + 4]], np.int32)))     # outside the pool: skipped
        assert kvc.kvc_pool_sync_status(pool) == kvc.KVC_ERR_BAD_BLOCK
    finally:
        pool.close()


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_allocator_copy_on_write_decode(kvc, dtype):
    """Tables from the host allocator drive the kernels: B forks A inside a
    partly filled block; before B's append the allocator maps a fresh block and
    kvc_copy_blocks copies the shared one; both then decode against the oracle."""
    L, H_Q, H, d, bs, N = 2, 16, 4, 128, 16, 32
    alloc = kvc.Allocator(N, bs)
    A = alloc.new_seq()
    alloc.reserve(A, 40)
    w = synth.make_workload("custom", B=2, H_Q=H_Q, H_KV=H, d_h=d, lens=[40, 40], L=L, dtype=dtype, seed=11)
    pool = kvc.kvc_pool_create(N, bs, L, H, d, kvc.KVC_FP8_E4M3 if dtype == "fp8" else kvc.KVC_BF16)
    try:
        pool.bytes_view().fill_(0x11)
        s = 1 if dtype == "fp8" else 2
        img = oracle.PoolImage(N, bs, L, H, d, s, fill=0x11)
        ctx = {l: (w.ctx_tokens(l, 0, 0, 0, 40), w.ctx_tokens(l, 1, 0, 0, 40)) for l in range(L)}
        tA, _ = alloc.block_tables([A], 3)
        for l in range(L):
            k, v = ctx[l]
            if dtype == "fp8":
                kvc.kvc_calibrate_fp8(pool, l, dev_bits(k), dev_bits(v))
                img.scales[l] = np.stack([oracle.fp8_scales(k), oracle.fp8_scales(v)])
            kvc.kvc_write_tokens(pool, l, dev_i32(tA), dev_i32([0]), dev_i32([0, 40]), dev_bits(k), dev_bits(v))
            img.write_tokens(l, tA, np.array([0], np.int32), np.array([0, 40], np.int64), k, v)
        alloc.commit(A, 40)
        B = alloc.fork(A, 40)                       # block 2 holds 8 of 16 positions: shared, partly filled
        cow = alloc.reserve(B, 1)
        assert len(cow) == 1 and cow[0][0] == int(tA[0, 2])
        kvc.kvc_copy_blocks(pool, dev_i32(np.array(cow, np.int32)))
        blk = img.bytes.size // (L * N)
        for l in range(L):
            o, n = cow[0]
            base = l * N * blk
            img.bytes[base + n * blk:base + (n + 1) * blk] = img.bytes[base + o * blk:base + (o + 1) * blk]
        assert alloc.reserve(A, 1) == []           # A's copy of the block is private again
        table, lens = alloc.block_tables([A, B], 3)
        assert table[0, 2] != table[1, 2] and lens.tolist() == [40, 40]
        bt, lp = dev_i32(table), dev_i32(lens)
        for l in range(L):
            q = w.q(l)
            kn, vn = w.kv_new(l, 0), w.kv_new(l, 1)
            out = torch.empty((2, H_Q, d), device="cuda")
            lse = torch.empty((2, H_Q), device="cuda")
            kvc.kvc_decode_step(pool, l, dev_bits(q), bt, lp, dev_bits(kn), dev_bits(vn), out, lse, scale=w.scale)
            torch.cuda.synchronize()
            assert kvc.kvc_pool_sync_status(pool) == kvc.KVC_OK
            img.append(l, table, lens, kn, vn)
            k, v = ctx[l]
            if dtype == "fp8":
                sk, sv = img.scales[l]
                kq, vq = oracle.quantize_e4m3(k, sk), oracle.quantize_e4m3(v, sv)
                nk, nv = oracle.quantize_e4m3(kn, sk), oracle.quantize_e4m3(vn, sv)
                scales = img.scales[l]
            else:
                kq, vq, nk, nv, scales = k, v, kn, vn, None
            K = np.concatenate([kq, nk[0:1], kq, nk[1:2]])
            V = np.concatenate([vq, nv[0:1], vq, nv[1:2]])
            ro, rl = oracle.decode(q, K, V, np.array([0, 41, 82]), np.array([41, 41]), H, scales=scales, scale=w.scale)
            check_attention(out, lse, ro, rl, dtype, f"copy-on-write layer {l}")
        alloc.commit(A, 1)
        alloc.commit(B, 1)
        n, first = first_mismatch(pool.bytes_view().cpu().numpy(), img.bytes)
        assert n == 0, f"{n} pool bytes differ, first at {first}"
    finally:
        pool.close()
        alloc.close()


@pytest.mark.parametrize("d_h", [64, 128])
@pytest.mark.parametrize("H_KV", [32, 16, 8])
def test_prefill_query_tiles(kvc, H_KV, d_h):
    """The query-tiled prefill kernel (bf16, groups of 1, 2, 4 query heads): chunks
    starting at 0 and inside a block, short and partial query tiles, several
    64-key stages, a row whose last block is part-filled; NaN in every unused
    pool byte; against the oracle."""
    H_Q = 32
    for q_start, n_q in ((0, 37), (45, 23), (200, 61), (1, 130), (333, 200)):
        total = q_start + n_q
        w = _custom(B=1, H_Q=H_Q, H_KV=H_KV, d_h=d_h, lens=[total], seed=q_start + n_q + H_KV)
        ld = layer_data(w, 0, with_step=False)
        g = GpuCase(kvc, w, fill_byte=0xFF)
        try:
            g.load_context(0, ld)
            qc = synth.normal_bf16(11, n_q, n_q * H_Q * d_h).reshape(n_q, H_Q, d_h)
            out = torch.full((n_q, H_Q, d_h), float("nan"), device="cuda")
            lse = torch.full((n_q, H_Q), float("nan"), device="cuda")
            kvc.kvc_prefill_attn(g.pool, 0, dev_bits(qc), g.bt[0], q_start, out, lse, scale=w.scale)
            torch.cuda.synchronize()
            assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
            ro, rl = oracle.prefill(qc, ld.k_ctx, ld.v_ctx, q_start, H_KV, scale=w.scale)
            check_attention(out, lse, ro, rl, "bf16", f"query tiles q_start={q_start} n_q={n_q}")
        finally:
            g.close()


@pytest.mark.parametrize("ppu", ["1", "3", "4", "8"])
@pytest.mark.parametrize("H_KV,dtype", [(8, "bf16"), (2, "bf16"), (32, "bf16"), (8, "fp8"), (8, "int4")])
def test_prefill_tiles(kvc, ppu, H_KV, dtype):
    """Causal prefill chunks whose CTAs serve several query positions (tail tile
    shorter, chunks starting inside a block) against the oracle."""
    H_Q, d = 32, 128
    if int(ppu) * (H_Q // H_KV) > 32:
        pytest.skip("more than 32 query columns per unit")
    os.environ["KVC_PREFILL_PPU"] = ppu
    try:
        for q_start, n_q in ((0, 37), (45, 23), (200, 61)):
            total = q_start + n_q
            w = _custom(B=1, H_Q=H_Q, H_KV=H_KV, d_h=d, lens=[total], dtype=dtype, seed=q_start + n_q)
            ld = layer_data(w, 0, with_step=False)
            g = GpuCase(kvc, w)
            try:
                g.load_context(0, ld)
                qc = synth.normal_bf16(7, n_q, n_q * H_Q * d).reshape(n_q, H_Q, d)
                out = torch.empty((n_q, H_Q, d), device="cuda")
                lse = torch.empty((n_q, H_Q), device="cuda")
                kvc.kvc_prefill_attn(g.pool, 0, dev_bits(qc), g.bt[0], q_start, out, lse, scale=w.scale)
                torch.cuda.synchronize()
                assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
                sc = None
                K, V = ld.k_ctx, ld.v_ctx
                if dtype != "bf16":   # the oracle's own calibration (the GPU's is checked against it)
                    cal = oracle.fp8_scales if dtype == "fp8" else oracle.int4_scales
                    sc = np.stack([cal(K), cal(V)]).astype(np.float32)
                    got = g.pool.scales_view()[0].cpu().numpy()
                    assert np.array_equal(got.view(np.uint32), sc.view(np.uint32)), "scales differ"
                    qz = oracle.quantize_e4m3 if dtype == "fp8" else oracle.quantize_int4
                    K, V = qz(K, sc[0]), qz(V, sc[1])
                ro, rl = oracle.prefill(qc, K, V, q_start, H_KV, scales=sc, scale=w.scale, kind=dtype)
                check_attention(out, lse, ro, rl, dtype, f"prefill ppu={ppu} q_start={q_start} n_q={n_q}")
            finally:
                g.close()
    finally:
        os.environ.pop("KVC_PREFILL_PPU", None)


@pytest.mark.parametrize("scale", [1.0, 0.37, 2.0 ** -6])
def test_int4_append_matches_codec_for_every_bf16(kvc, scale):
    """Every bf16 bit pattern written through an int4 pool: the stored nibble is
    the oracle's rint(fp32(x) / scale) clamped to [-7, 7] (+8), NaN -> 8, and the
    two channels of a byte land in its low and high nibble."""
    H, d = 1, 128
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    n_tok = 65536 // (H * d)
    N = n_tok // 16
    pool = kvc.kvc_pool_create(N, 16, 1, H, d, kvc.KVC_INT4)
    try:
        pool.bytes_view().fill_(0)
        s = torch.full((H, d), scale, dtype=torch.float32, device="cuda")
        kvc.kvc_pool_set_scales(pool, 0, s, s)
        x = bits.reshape(n_tok, H, d)
        bt = np.arange(N, dtype=np.int32).reshape(1, N)
        kvc.kvc_write_tokens(pool, 0, dev_i32(bt), dev_i32([0]), dev_i32([0, n_tok]), dev_bits(x), dev_bits(x))
        torch.cuda.synchronize()
        img = oracle.PoolImage(N, 16, 1, H, d, "int4")
        img.scales[0] = np.float32(scale)
        img.write_tokens(0, bt, np.array([0], np.int32), np.array([0, n_tok], np.int64), x, x)
        n, first = first_mismatch(pool.bytes_view().cpu().numpy(), img.bytes)
        assert n == 0, f"{n} bytes differ, first at {first}"
    finally:
        pool.close()
