"""The seeded input generators: determinism, random access, distribution, recipes."""
import math

import numpy as np
import pytest

import synth


def test_counter_based_random_access():
    a = synth.normal_bf16(0, 5, 1000)
    b = synth.normal_bf16(0, 5, 300, offset=700)
    assert np.array_equal(a[700:], b)
    assert np.array_equal(a, synth.normal_bf16(0, 5, 1000))
    assert not np.array_equal(a, synth.normal_bf16(1, 5, 1000))
    assert not np.array_equal(a, synth.normal_bf16(0, 6, 1000))


def test_normal_moments():
    x = synth.normal_f64(0, 1, 200_000)
    assert abs(x.mean()) < 0.01 and abs(x.var() - 1) < 0.01
    assert abs((x > 1.959964).mean() - 0.025) < 0.002


def test_bf16_rounding_nearest_even():
    x = synth.normal_f64(2, 3, 20000) * np.exp(synth.normal_f64(2, 4, 20000) * 5)
    for v in x:
        bits = synth.lib().synth_bf16_from_double(float(v))
        r = float(synth.bf16_bits_to_f32(np.array([bits], np.uint16))[0])
        e = math.frexp(abs(v))[1] - 1
        ulp = 2.0 ** (e - 7)
        assert abs(r - v) <= ulp / 2
        if abs(r - v) == ulp / 2:
            assert bits & 1 == 0
    # ties: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> even (1.0)
    assert synth.lib().synth_bf16_from_double(1 + 2 ** -8) == 0x3F80
    assert synth.lib().synth_bf16_from_double(1 + 3 * 2 ** -8) == 0x3F82


def test_permutation_is_permutation():
    p = synth.permutation(0, 9, 16416)
    assert np.array_equal(np.sort(p), np.arange(16416))
    assert not np.array_equal(p, np.arange(16416))


@pytest.mark.parametrize("name", ["tiny", "llama_gqa", "ragged_prefix", "sweep_hkv1_fp8", "full_pool"])
def test_workload_tables_are_disjoint_and_sized(name):
    w = synth.make_workload(name, seed=0)
    bt = w.block_tables
    rows = bt.shape[0]
    used = []
    for r in range(rows):
        n = w.row_len(r) + (0 if (w.prefill and r == w.prefill.seq) else 1)
        nb = -(-n // w.bs)
        assert np.all(bt[r, :nb] >= 0) and np.all(bt[r, nb:] == -1)
        used.append(bt[r, w.shared_prefix // w.bs:nb])
    used = np.concatenate(used)
    shared = bt[0, :w.shared_prefix // w.bs]
    assert len(np.unique(used)) == len(used)                       # private blocks never alias
    assert not np.intersect1d(used, shared).size
    assert np.all(bt[bt >= 0] < w.num_blocks)
    assert len(used) + len(shared) <= w.num_blocks


def test_workload_shapes():
    w = synth.make_workload("tiny")
    assert (w.B, w.H_Q, w.H_KV, w.d_h, w.num_blocks) == (4, 8, 2, 64, 128)
    assert np.all((w.lens_pre >= 1) & (w.lens_pre <= 256))
    w = synth.make_workload("llama_gqa")
    assert w.num_blocks == 32 * 513 and w.kv_bytes_read() == 1_073_872_896
    w = synth.make_workload("full_pool")
    assert w.num_blocks == 16392 and w.L == 32
    w = synth.make_workload("ragged_prefix")
    assert w.B == 64 and np.all(w.lens_pre >= 1200) and np.all(w.lens_pre <= 32768)
    assert w.prefill.total == 1800 and w.block_tables.shape[0] == 65
    # 1800 tokens need 113 blocks: 75 shared + 38 private
    assert int((w.block_tables[64] >= 0).sum()) == 113


def test_ctx_tokens_slices_and_shared_prefix():
    w = synth.make_workload("ragged_prefix")
    a = w.ctx_tokens(0, 0, 3, 0, 1300)
    b = w.ctx_tokens(0, 0, 3, 1100, 1300)
    assert np.array_equal(a[1100:], b)
    c = w.ctx_tokens(0, 0, 9, 0, 1200)
    assert np.array_equal(a[:1200], c)              # the shared prefix is the same for every row
    assert not np.array_equal(a[1200:1300], w.ctx_tokens(0, 0, 9, 1200, 1300))
