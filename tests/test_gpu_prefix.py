"""Prefix identity through the GPU path.

"KV cache: Generation state, latency, and allocation" 21.4 (a block is
reused when its whole token prefix matches), "KV Cache Explained", "Prefix
reuse saves prefill, while decode still needs the history", and the
xf_kv_cache page, "End-to-end flow" (a 1 800-token request whose first 1 200
tokens, 75 blocks of 16, are found resident; only the 600 new tokens are
prefilled, and decode reads the whole history).

The host block allocator (C ABI) publishes a request's 1 200-token prompt and
matches later requests against it; the tables it hands out drive the
token writes, the fused decode step and a 600-query prefill chunk.  The
oracle's allocator model replays the same operations (tables, reference
counts, counts), the oracle's pool image receives the same writes (every pool
byte compared), and the oracle's attention runs over each request's logical
history (shared prompt + private tokens + the appended one).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from harness import check_attention, dev_bits, dev_i32, first_mismatch, scale_of
from oracle.allocator import BlockAllocator

pytestmark = pytest.mark.gpu

H_Q, H_KV, D, BS = 32, 8, 128, 16
N_BLOCKS, MAX_BLOCKS = 600, 160
SHARED = 1200          # 75 full blocks
SEED = 41


def _kv(stream, n):
    return synth.normal_bf16(SEED, stream, n * H_KV * D).reshape(n, H_KV, D)


def _ids(stream, n):
    return (synth.u64(SEED, stream, n) % 32000).astype(np.int32)


def test_published_prefix_drives_decode_and_prefill(kvc):
    scale = scale_of(D)
    perm = synth.permutation(SEED, 1, N_BLOCKS)
    alloc = kvc.Allocator(N_BLOCKS, BS, free_order=perm, retain_cached=True)
    model = BlockAllocator(N_BLOCKS, BS, free_order=perm, retain_cached=True)
    pool = kvc.kvc_pool_create(N_BLOCKS, BS, 1, H_KV, D, kvc.KVC_BF16)
    pool.bytes_view().fill_(0xFF)
    img = oracle.PoolImage(N_BLOCKS, BS, 1, H_KV, D, 2, fill=0xFF)
    try:
        def write(sc, sm, start, k, v):
            """Reserve, write positions [start, start + n) through the allocator's table, commit."""
            n = len(k)
            assert alloc.reserve(sc, n) == [] and model.reserve(sm, n) == []
            table, _ = alloc.block_tables([sc], MAX_BLOCKS)
            assert table[0].tolist() == model.table(sm, MAX_BLOCKS)
            kvc.kvc_write_tokens(pool, 0, dev_i32(table), dev_i32([start]), dev_i32([0, n]), dev_bits(k), dev_bits(v))
            assert img.write_tokens(0, table, np.array([start], np.int32), np.array([0, n], np.int64), k, v) == oracle.OK
            alloc.commit(sc, n)
            model.commit(sm, n)

        # request A writes and publishes the shared prompt
        prompt = _ids(2, SHARED)
        a, am = alloc.new_seq(), model.new_seq()
        kA, vA = _kv(10, SHARED), _kv(11, SHARED)
        write(a, am, 0, kA, vA)
        alloc.publish(a, prompt)
        model.publish(am, prompt)
        history = {a: (kA, vA)}

        # three requests with the same prompt and private continuations: matched, then their own tokens
        seqs = [(a, am)]
        for i, n_own in enumerate([37, 300, 16]):
            toks = np.concatenate([prompt, _ids(20 + i, n_own)])
            (r, hit), (rm, hit_m) = alloc.match(toks), model.match(toks)
            assert hit == hit_m == SHARED
            k_own, v_own = _kv(30 + i, n_own), _kv(40 + i, n_own)
            write(r, rm, SHARED, k_own, v_own)
            history[r] = (np.concatenate([kA, k_own]), np.concatenate([vA, v_own]))
            seqs.append((r, rm))
        prompt_blocks = alloc.block_tables([a], MAX_BLOCKS)[0][0][:SHARED // BS]
        for blk in prompt_blocks:
            assert alloc.refcount(int(blk)) == model.ref[int(blk)] == 4

        # one decode step over all four: a position each, the fused append + attention
        for sc, sm in seqs:
            assert alloc.reserve(sc, 1) == [] and model.reserve(sm, 1) == []
        table, lens = alloc.block_tables([sc for sc, _ in seqs], MAX_BLOCKS)
        for (sc, sm), row in zip(seqs, table):
            assert row.tolist() == model.table(sm, MAX_BLOCKS)
        B = len(seqs)
        q = synth.normal_bf16(SEED, 50, B * H_Q * D).reshape(B, H_Q, D)
        k_new, v_new = _kv(51, B), _kv(52, B)
        out = torch.empty((B, H_Q, D), device="cuda")
        lse = torch.empty((B, H_Q), device="cuda")
        kvc.kvc_decode_step(pool, 0, dev_bits(q), dev_i32(table), dev_i32(lens), dev_bits(k_new), dev_bits(v_new),
                            out, lse, scale=scale)
        assert img.append(0, table, lens, k_new, v_new) == oracle.OK
        for sc, sm in seqs:
            alloc.commit(sc, 1)
            model.commit(sm, 1)
        torch.cuda.synchronize()
        assert kvc.kvc_pool_sync_status(pool) == kvc.KVC_OK
        Ks = [np.concatenate([history[sc][0], k_new[b:b + 1]]) for b, (sc, _) in enumerate(seqs)]
        Vs = [np.concatenate([history[sc][1], v_new[b:b + 1]]) for b, (sc, _) in enumerate(seqs)]
        cu = np.concatenate([[0], np.cumsum([len(k) for k in Ks])]).astype(np.int64)
        ro, rl = oracle.decode(q, np.concatenate(Ks), np.concatenate(Vs), cu, lens.astype(np.int64) + 1, H_KV,
                               scale=scale)
        check_attention(out, lse, ro, rl, "bf16", "decode over matched prefixes")

        # the 1 800-token request: 1 200 matched, its 600 new tokens written and prefilled causally
        toks = np.concatenate([prompt, _ids(60, 600)])
        (r4, hit), (r4m, hit_m) = alloc.match(toks), model.match(toks)
        assert hit == hit_m == SHARED
        kc, vc = _kv(61, 600), _kv(62, 600)
        write(r4, r4m, SHARED, kc, vc)
        row = alloc.block_tables([r4], MAX_BLOCKS)[0][0]
        qc = synth.normal_bf16(SEED, 63, 600 * H_Q * D).reshape(600, H_Q, D)
        o2 = torch.empty((600, H_Q, D), device="cuda")
        l2 = torch.empty((600, H_Q), device="cuda")
        kvc.kvc_prefill_attn(pool, 0, dev_bits(qc), dev_i32(row), SHARED, o2, l2, scale=scale)
        torch.cuda.synchronize()
        assert kvc.kvc_pool_sync_status(pool) == kvc.KVC_OK
        ro2, rl2 = oracle.prefill(qc, np.concatenate([kA, kc]), np.concatenate([vA, vc]), SHARED, H_KV, scale=scale)
        check_attention(o2, l2, ro2, rl2, "bf16", "prefill chunk over the matched prefix")
        for blk in prompt_blocks:
            assert alloc.refcount(int(blk)) == model.ref[int(blk)] == 5

        # every pool byte, shared and private blocks and untouched ones
        n, first = first_mismatch(pool.bytes_view().cpu().numpy(), img.bytes)
        assert n == 0, f"{n} pool bytes differ, first at {first}"

        # releases drop the prompt blocks' references; the published blocks stay matchable
        for sc, sm in seqs[1:]:
            alloc.release(sc)
            model.release(sm)
        for blk in prompt_blocks:
            assert alloc.refcount(int(blk)) == model.ref[int(blk)] == 2
        assert alloc.counts() == model.counts()
    finally:
        pool.close()
        alloc.close()
