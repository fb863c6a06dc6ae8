"""Expired waits on the GPU: bounded mbarrier waits report KVC_ERR_TIMEOUT.

Every wait in the decode and prefill kernels is bounded (2 s of %globaltimer);
on expiry the kernel records KVC_ERR_TIMEOUT in the pool's error word, lets
its own copies drain, frees its tensor memory and returns.  The test hook
KVC_TEST_STALL makes the copy producers issue no load and never arrive, so the
first wait of every consumer runs out -- nothing is in flight, nothing faults.
Each case checks the status, then runs the same call without the hook on the
same pool and compares it with the oracle: the context and the pool stay
usable.  Cases: the split kernel (bf16 GQA and e4m3), the tensor-memory MQA
kernels (bf16 and e4m3) through the fused step, and the tensor-memory prefill
kernel.
"""
import os

import pytest
import torch

import oracle
import synth
from harness import GpuCase, OracleCase, check_attention, dev_bits, first_mismatch, layer_data

pytestmark = pytest.mark.gpu


def _stalled(fn):
    os.environ["KVC_TEST_STALL"] = "1"
    try:
        fn()
        torch.cuda.synchronize()
    finally:
        os.environ.pop("KVC_TEST_STALL", None)


DECODE_CASES = [("bf16", 8, [300, 40]), ("fp8", 8, [500, 17]), ("bf16", 1, [700, 129]), ("fp8", 1, [900, 33])]


@pytest.mark.parametrize("dtype,H_KV,lens", DECODE_CASES,
                         ids=[f"{c[0]}-hkv{c[1]}" for c in DECODE_CASES])
def test_expired_waits_in_the_decode_step(kvc, dtype, H_KV, lens):
    w = synth.make_workload("custom", B=len(lens), H_Q=32, H_KV=H_KV, d_h=128, lens=lens, dtype=dtype, seed=7)
    g = GpuCase(kvc, w, fill_byte=0xFF)
    try:
        ld = layer_data(w, 0)
        g.load_context(0, ld)
        q, k_new, v_new = g.step_inputs(ld)
        out = torch.full((w.B, w.H_Q, w.d_h), float("nan"), device="cuda")
        lse = torch.full((w.B, w.H_Q), float("nan"), device="cuda")
        step = lambda: kvc.kvc_decode_step(g.pool, 0, q, g.bt_dec, g.lens_pre, k_new, v_new, out, lse,
                                           scale=w.scale)
        _stalled(step)
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_ERR_TIMEOUT
        step()                                  # the hook off: the same call on the same pool
        torch.cuda.synchronize()
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
        ref = OracleCase(w, fill_byte=0xFF).run_layer(ld)
        n, first = first_mismatch(g.layer_bytes(0), ref["image"].bytes)
        assert n == 0, f"{n} pool bytes differ, first at {first}"
        check_attention(out, lse, ref["out"], ref["lse"], dtype, f"after an expired wait {dtype} H_KV={H_KV}")
    finally:
        g.close()


def test_expired_waits_in_the_prefill_chunk(kvc):
    q_start, n_q, H_Q, H_KV, d_h = 200, 150, 32, 8, 128
    w = synth.make_workload("custom", B=1, H_Q=H_Q, H_KV=H_KV, d_h=d_h, lens=[q_start + n_q], seed=11)
    ld = layer_data(w, 0, with_step=False)
    g = GpuCase(kvc, w, fill_byte=0xFF)
    try:
        g.load_context(0, ld)
        qc = synth.normal_bf16(19, n_q, n_q * H_Q * d_h).reshape(n_q, H_Q, d_h)
        out = torch.full((n_q, H_Q, d_h), float("nan"), device="cuda")
        lse = torch.full((n_q, H_Q), float("nan"), device="cuda")
        call = lambda: kvc.kvc_prefill_attn(g.pool, 0, dev_bits(qc), g.bt[0], q_start, out, lse, scale=w.scale)
        _stalled(call)
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_ERR_TIMEOUT
        call()
        torch.cuda.synchronize()
        assert kvc.kvc_pool_sync_status(g.pool) == kvc.KVC_OK
        ro, rl = oracle.prefill(qc, ld.k_ctx, ld.v_ctx, q_start, H_KV, scale=w.scale)
        check_attention(out, lse, ro, rl, "bf16", "prefill after an expired wait")
    finally:
        g.close()
