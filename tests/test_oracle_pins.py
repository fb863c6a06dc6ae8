"""Pins of the CPU oracle to facts outside itself (no GPU).

Each test checks the oracle against something the pages or the mathematics fix:
printed worked-example values (tests/golden/), the block mapping of Table 21.1,
an independent library routine (torch's float64 attention and its
float8_e4m3fn conversion), brute force, closed forms and invariants.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GIB = 1024 ** 3


# ---------------------------------------------------------------- Eq. 21.2 / 21.3
def _golden_rows(name):
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            yield line


def _page_cases():
    rows = []
    for line in _golden_rows("page_values.txt"):
        fn, args, expected, cite = [x.strip() for x in line.split("|", 3)]
        rows.append(pytest.param(fn, [int(a) for a in args.split()], float(expected), id=f"{fn}:{args}"))
    return rows


LLAMA = dict(L=32, H_KV=8, d_h=128, s=2)   # the Llama-3.1-8B-style shape of "KV Cache Explained"


@pytest.mark.parametrize("fn,args,expected", _page_cases())
def test_page_values(fn, args, expected):
    if fn == "kv_bytes":
        got = oracle.kv_bytes(*args)
    elif fn == "growth":
        got = oracle.kv_bytes_growth(*args)
    elif fn == "gib":
        got = oracle.kv_bytes(*args) / GIB
    elif fn == "values_per_tensor":
        L, B, H, T, d, s = args
        got = oracle.kv_bytes(L, B, H, T, d, s) / (2 * s)
    elif fn == "blocks":
        tokens, bs = args
        got = tokens // bs
    elif fn == "pool_blocks":
        pool_gib, bs = args
        got = pool_gib * GIB // oracle.kv_bytes(LLAMA["L"], 1, LLAMA["H_KV"], bs, LLAMA["d_h"], LLAMA["s"])
    elif fn == "shared_gib":
        prefix, suffix, nreq = args
        got = (oracle.kv_bytes(32, 1, 8, prefix, 128, 2) + oracle.kv_bytes(32, nreq, 8, suffix, 128, 2)) / GIB
    elif fn == "transfer_s":
        gib, gbs = args
        got = round(oracle.kv_bytes(32, 1, 8, 32768, 128, 2) * gib / 4 / (gbs * 1e9), 2)
    else:
        raise AssertionError(fn)
    assert got == expected


def test_eq_21_3_is_growth_of_eq_21_2():
    # Eq. 21.3 is the difference of Eq. 21.2 at T+1 and T, for any shape
    for (L, B, H, d, s) in [(2, 1, 4, 8, 2), (32, 8, 8, 128, 2), (1, 3, 5, 7, 1)]:
        for T in (0, 1, 17, 8192):
            assert oracle.kv_bytes(L, B, H, T + 1, d, s) - oracle.kv_bytes(L, B, H, T, d, s) == \
                oracle.kv_bytes_growth(L, B, H, d, s)


def test_kv_bytes_overflow_and_negative():
    assert oracle.kv_bytes(2**20, 2**20, 2**20, 2**20, 1, 1) == 2**64 - 1
    assert oracle.kv_bytes(-1, 1, 1, 1, 1, 1) == 2**64 - 1
    assert oracle.kv_bytes(32, 0, 8, 100, 128, 2) == 0


# ---------------------------------------------------------------- Table 21.1
def _table_fixture():
    bs = N = None
    tables, lens, steps = {}, {}, []
    for line in _golden_rows("table_21_1.txt"):
        w = line.split()
        if w[0] == "block_size":
            bs = int(w[1])
        elif w[0] == "pool_blocks":
            N = int(w[1])
        elif w[0] == "table":
            tables[w[1]] = [int(x) for x in w[2:]]
        elif w[0] == "len":
            lens[w[1]] = int(w[2])
        else:
            steps.append(w)
    return bs, N, tables, lens, steps


def test_table_21_1_address_translation():
    bs, N, tables, _, steps = _table_fixture()
    for w in steps:
        if w[0] != "locate":
            continue
        row = np.array(tables[w[1]], dtype=np.int32)
        st, phys, slot = oracle.locate(row, int(w[2]), bs, N)
        if w[4] == "range":
            assert st == oracle.ERR_RANGE
        else:
            assert st == oracle.OK and (phys, slot) == (int(w[4]), int(w[5]))


def test_pool_layout_structure():
    """The pool image's layout (the library's documented format, not the pages'):
    every element has its own offset and the offsets fill the allocation; the keys
    then the values of one (layer, block, head) form one contiguous run of
    2 * bs * d_h elements, slot-major; the heads of a block follow each other; a
    layer's region is N * H_KV * 2 * bs * d_h elements, so one block id names the same
    block in every layer ("KV Cache Explained", "Why PagedAttention allocates KV in
    blocks": 2 MiB per 16-token block across 32 layers for 8 KV heads of width 128
    in bf16)."""
    L, N, H, bs, d = 3, 5, 4, 4, 8
    img = oracle.PoolImage(N, bs, L, H, d, 2)
    # visiting (layer, block, head, K|V, slot, channel) in that nesting order walks the
    # allocation element by element: 0, 1, 2, ... -- which is every property above at once
    offs = [img.offset(l, p, kv, h, slot, c)
            for l in range(L) for p in range(N) for h in range(H)
            for kv in range(2) for slot in range(bs) for c in range(d)]
    assert offs == list(range(L * N * H * 2 * bs * d))
    llama = oracle.PoolImage(1, 16, 32, 8, 128, 2)
    per_block_all_layers = 32 * (llama.offset(0, 1, 0, 0, 0, 0) - llama.offset(0, 0, 0, 0, 0, 0)) * 2
    assert per_block_all_layers == 2 * 2**20


def test_table_21_1_appends_through_pool_image():
    """Replay steps 1-2 with distinct token values and check where the bytes land."""
    bs, N, tables, lens, steps = _table_fixture()
    H, d = 1, 2
    img = oracle.PoolImage(N, bs, 1, H, d, 2, fill=0xEE)
    rows = {"A": list(tables["A"]), "B": list(tables["B"])}
    width = 3

    def bt():
        out = np.full((2, width), -1, dtype=np.int32)
        for i, r in enumerate(("A", "B")):
            out[i, :len(rows[r])] = rows[r]
        return out

    before_B = None
    for w in steps:
        if w[0] == "extend":
            rows[w[1]].append(int(w[2]))
        elif w[0] == "append":
            pos, phys, slot = int(w[2]), int(w[4]), int(w[5])
            k = np.array([[[1000 + pos, 2000 + pos]]], dtype=np.uint16)
            v = np.array([[[3000 + pos, 4000 + pos]]], dtype=np.uint16)
            if before_B is None:
                before_B = img.gather(0, bt()[1], 4)
            st = img.write_tokens(0, bt()[:1], np.array([pos], dtype=np.int32),
                                  np.array([0, 1], dtype=np.int64), k, v)
            assert st == oracle.OK
            for kv, src in ((0, k), (1, v)):
                for c in range(d):
                    off = img.offset(0, phys, kv, 0, slot, c) * 2
                    val = int(img.bytes[off]) | (int(img.bytes[off + 1]) << 8)
                    assert val == int(src[0, 0, c])
    # B's block is untouched by A's appends (Table 21.1 step 4: B still owns block 9)
    assert all(np.array_equal(a, b) for a, b in zip(before_B[1:], img.gather(0, bt()[1], 4)[1:]))
    # A now reads positions 6, 7, 8 back in logical order through [7, 2, 5]
    st, kA, vA = img.gather(0, bt()[0], 9)
    assert st == oracle.OK
    assert [int(kA[t, 0, 0]) for t in (6, 7, 8)] == [1006, 1007, 1008]


def test_write_gather_roundtrip_random_tables():
    """Writing through random tables and gathering back returns the logical list
    bit for bit; every byte outside the written slots keeps its fill."""
    rng = np.random.default_rng(7)
    for bs, H, d, s in [(16, 2, 8, 2), (4, 3, 4, 2), (16, 2, 8, 1), (8, 1, 16, 1)]:
        B = 5
        lens = rng.integers(1, 60, size=B)
        nb = -(-lens // bs)
        N = int(nb.sum()) + 7
        perm = rng.permutation(N).astype(np.int32)
        mb = int(nb.max()) + 2
        bt = np.full((B, mb), -1, dtype=np.int32)
        cur = 0
        for b in range(B):
            bt[b, :nb[b]] = perm[cur:cur + nb[b]]
            cur += nb[b]
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        k = rng.integers(0, 2**16, size=(int(cu[-1]), H, d), dtype=np.uint16)
        v = rng.integers(0, 2**16, size=(int(cu[-1]), H, d), dtype=np.uint16)
        if s == 1:   # finite bf16 inputs only (fp8 path quantises)
            k = synth.normal_bf16(1, 1, k.size).reshape(k.shape)
            v = synth.normal_bf16(1, 2, v.size).reshape(v.shape)
        img = oracle.PoolImage(N, bs, 1, H, d, s, fill=0x5A)
        if s == 1:
            img.scales[0] = np.float32(0.01)
        assert img.write_tokens(0, bt, np.zeros(B, np.int32), cu, k, v) == oracle.OK
        written = 0
        for b in range(B):
            st, kb, vb = img.gather(0, bt[b], int(lens[b]))
            assert st == oracle.OK
            if s == 2:
                assert np.array_equal(kb, k[cu[b]:cu[b + 1]]) and np.array_equal(vb, v[cu[b]:cu[b + 1]])
            else:
                exp_k = np.vectorize(lambda x: oracle.e4m3_encode(np.float32(synth.bf16_bits_to_f32(np.array([x], np.uint16))[0] / np.float32(0.01))))(k[cu[b]:cu[b + 1]])
                assert np.array_equal(kb, exp_k.astype(np.uint8))
            written += 2 * int(lens[b]) * H * d * s
        untouched = img.bytes == 0x5A
        assert int((~untouched).sum()) <= written
        # a permutation of the physical blocks (tables rewritten) gives the same logical lists
        remap = rng.permutation(N).astype(np.int32)
        bt2 = np.where(bt >= 0, remap[np.maximum(bt, 0)], -1).astype(np.int32)
        img2 = oracle.PoolImage(N, bs, 1, H, d, s, fill=0x00)
        img2.scales[:] = img.scales
        img2.write_tokens(0, bt2, np.zeros(B, np.int32), cu, k, v)
        for b in range(B):
            a = img.gather(0, bt[b], int(lens[b]))
            c = img2.gather(0, bt2[b], int(lens[b]))
            assert np.array_equal(a[1], c[1]) and np.array_equal(a[2], c[2])


def test_write_errors_skip_only_the_bad_token():
    img = oracle.PoolImage(4, 4, 1, 1, 2, 2, fill=0)
    bt = np.array([[0, -1, 2], [1, 3, 9]], dtype=np.int32)     # -1 unallocated, 9 outside the pool
    k = np.arange(1, 1 + 12 * 2, dtype=np.uint16).reshape(12, 1, 2)
    cu = np.array([0, 6, 12], dtype=np.int64)
    st = img.write_tokens(0, bt, np.array([2, 6], np.int32), cu, k, k)
    assert st == oracle.ERR_BAD_BLOCK
    # sequence 0: positions 2,3 valid (block 0), 4..7 in block -1 skipped
    assert img.gather(0, bt[0], 4)[0] == oracle.OK
    assert oracle.locate(bt[0], 4, 4, 4)[0] == oracle.ERR_BAD_BLOCK
    assert oracle.locate(bt[1], 12, 4, 4)[0] == oracle.ERR_RANGE
    assert oracle.locate(bt[1], 8, 4, 4)[0] == oracle.ERR_BAD_BLOCK


# ---------------------------------------------------------------- e4m3 codec
def _torch_e4m3(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_decode(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours)) and set(codes[nan]) == {0x7F, 0xFF}
    assert np.array_equal(ref[~nan], ours[~nan])
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_values_are_exact_in_f16():
    """Every finite e4m3 value is an f16 value (4 significant bits, exponents 2^-9 .. 2^8 inside f16's
    2^-24 .. 2^15), so widening the codes to f16 before a tensor-core product loses nothing."""
    vals = np.array([oracle.e4m3_decode(c) for c in range(256) if c & 0x7F != 0x7F])
    assert len(vals) == 254 and np.all(np.isfinite(vals))
    assert np.array_equal(vals.astype(np.float16).astype(np.float64), vals)


def test_e4m3_encode_every_bf16_vs_torch():
    bits = np.arange(65536, dtype=np.uint32)
    x = ((bits << 16).astype(np.uint32)).view(np.float32)
    ok = np.isfinite(x) & (np.abs(x) <= 464.0)        # torch turns > 464 into NaN, not 448
    enc = np.array([oracle.e4m3_encode(float(v)) for v in x[ok]], dtype=np.uint8)
    assert np.array_equal(enc, _torch_e4m3(x[ok]))
    big = x[np.isfinite(x) & (np.abs(x) > 464.0)]
    sat = np.array([oracle.e4m3_encode(float(v)) for v in big], dtype=np.uint8)
    assert np.all(sat == np.where(big > 0, 0x7E, 0xFE))
    assert oracle.e4m3_encode(float("inf")) == 0x7E and oracle.e4m3_encode(float("-inf")) == 0xFE


def test_e4m3_encode_quotients_and_ties_vs_bruteforce():
    """fp32 quotients x/s (the append's input) and exact midpoints between codes:
    the code must be the nearest finite one, ties to the even mantissa."""
    finite = np.array([oracle.e4m3_decode(c) for c in range(0x7F)])   # positive codes 0..0x7E
    mids = (finite[:-1] + finite[1:]) / 2
    xs = list(mids.astype(np.float32)) + list(-mids.astype(np.float32))
    b = synth.normal_bf16(3, 1, 4000)
    for s in (np.float32(1.0), np.float32(1 / 448), np.float32(4.25 / 448), np.float32(2.0 ** -12)):
        xs += list(synth.bf16_bits_to_f32(b) / s)
    for x in xs:
        x = np.float32(x)
        a = abs(float(x))
        if a >= 448:
            want = 0x7E
        else:
            dist = np.abs(finite - a)
            best = np.flatnonzero(dist == dist.min())
            want = int(best[0]) if len(best) == 1 else int([c for c in best if c % 2 == 0][0])
        if x < 0 or (x == 0 and math.copysign(1, x) < 0):
            want |= 0x80
        assert oracle.e4m3_encode(float(x)) == want, (x, want)


def test_fp8_scales_definition():
    x = synth.normal_bf16(5, 9, 64 * 2 * 8).reshape(64, 2, 8)
    sc = oracle.fp8_scales(x)
    xf = synth.bf16_bits_to_f32(x)
    assert np.array_equal(sc, (np.abs(xf).max(axis=0) / np.float32(448)).astype(np.float32))
    assert np.array_equal(oracle.fp8_scales(np.zeros((3, 1, 2), np.uint16)), np.ones((1, 2), np.float32))


# ---------------------------------------------------------------- attention
def _torch_causal_last_row(q_last, Kd, Vd, H_Q, scale, rng):
    """Full causal attention recomputed from scratch (no cache) over n positions
    with float64 library routines; returns the last position's output and lse."""
    n, H_KV, d = Kd.shape
    Q = torch.from_numpy(rng.standard_normal((n, H_Q, d)))
    Q[-1] = torch.from_numpy(q_last)
    qh = Q.permute(1, 0, 2).unsqueeze(0)                # [1, H_Q, n, d]
    kh = torch.from_numpy(Kd).permute(1, 0, 2).unsqueeze(0)
    vh = torch.from_numpy(Vd).permute(1, 0, 2).unsqueeze(0)
    out = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, is_causal=True, scale=scale,
                                                           enable_gqa=True)
    g = H_Q // H_KV
    scores = torch.einsum("hd,htd->ht", qh[0, :, -1], kh[0].repeat_interleave(g, dim=0)) * scale
    lse = torch.logsumexp(scores, dim=-1)
    return out[0, :, -1].numpy(), lse.numpy()


def _dequant(stored, scales_hc=None):
    if stored.dtype == np.uint16:
        return synth.bf16_bits_to_f32(stored).astype(np.float64)
    dec = np.array([oracle.e4m3_decode(c) for c in range(256)])
    return dec[stored] * scales_hc.astype(np.float64)[None]


@pytest.mark.parametrize("H_Q,H_KV,d,lens", [(8, 2, 16, [1, 2, 17, 40]), (4, 4, 8, [3, 16, 33]),
                                              (8, 1, 16, [5, 31, 32]), (6, 3, 8, [1, 9])])
def test_decode_equals_full_recompute_bf16(H_Q, H_KV, d, lens):
    rng = np.random.default_rng(H_Q * 100 + d)
    B = len(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    K = synth.normal_bf16(11, H_Q, int(cu[-1]) * H_KV * d).reshape(-1, H_KV, d)
    V = synth.normal_bf16(12, H_Q, int(cu[-1]) * H_KV * d).reshape(-1, H_KV, d)
    q = synth.normal_bf16(13, H_Q, B * H_Q * d).reshape(B, H_Q, d)
    scale = float(np.float32(1 / math.sqrt(d)))
    out, lse = oracle.decode(q, K, V, cu, np.array(lens), H_KV, scale=scale)
    for b in range(B):
        Kd, Vd = _dequant(K[cu[b]:cu[b + 1]]), _dequant(V[cu[b]:cu[b + 1]])
        ro, rl = _torch_causal_last_row(synth.bf16_bits_to_f32(q[b]).astype(np.float64), Kd, Vd, H_Q, scale, rng)
        np.testing.assert_allclose(out[b], ro, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b], rl, rtol=0, atol=1e-12)


def test_decode_equals_full_recompute_fp8():
    rng = np.random.default_rng(3)
    H_Q, H_KV, d, lens = 8, 2, 16, [1, 7, 24]
    B = len(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    Kb = synth.normal_bf16(21, 1, int(cu[-1]) * H_KV * d).reshape(-1, H_KV, d)
    Vb = synth.normal_bf16(21, 2, int(cu[-1]) * H_KV * d).reshape(-1, H_KV, d)
    sc = np.stack([oracle.fp8_scales(Kb), oracle.fp8_scales(Vb)])
    enc = np.vectorize(lambda x: oracle.e4m3_encode(float(x)))
    K = enc(synth.bf16_bits_to_f32(Kb) / sc[0][None]).astype(np.uint8)
    V = enc(synth.bf16_bits_to_f32(Vb) / sc[1][None]).astype(np.uint8)
    q = synth.normal_bf16(22, 1, B * H_Q * d).reshape(B, H_Q, d)
    scale = 0.25
    out, lse = oracle.decode(q, K, V, cu, np.array(lens), H_KV, scales=sc, scale=scale)
    for b in range(B):
        Kd, Vd = _dequant(K[cu[b]:cu[b + 1]], sc[0]), _dequant(V[cu[b]:cu[b + 1]], sc[1])
        ro, rl = _torch_causal_last_row(synth.bf16_bits_to_f32(q[b]).astype(np.float64), Kd, Vd, H_Q, scale, rng)
        np.testing.assert_allclose(out[b], ro, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b], rl, rtol=0, atol=1e-12)


def test_decode_closed_forms():
    H_Q, H_KV, d = 4, 2, 8
    q = synth.normal_bf16(31, 0, H_Q * d).reshape(1, H_Q, d)
    K = synth.normal_bf16(31, 1, 50 * H_KV * d).reshape(50, H_KV, d)
    V = synth.normal_bf16(31, 2, 50 * H_KV * d).reshape(50, H_KV, d)
    scale = 0.3
    qd = synth.bf16_bits_to_f32(q[0]).astype(np.float64)
    # one position: the output is that value exactly, lse its scaled score
    out, lse = oracle.decode(q, K, V, np.array([0, 1]), np.array([1]), H_KV, scale=scale)
    for hq in range(H_Q):
        h = hq // (H_Q // H_KV)
        assert np.array_equal(out[0, hq], synth.bf16_bits_to_f32(V[0, h]).astype(np.float64))
        assert lse[0, hq] == pytest.approx(scale * qd[hq] @ synth.bf16_bits_to_f32(K[0, h]), abs=1e-12)
    # every key equal: uniform weights, the output is the mean value, lse = x + ln n
    Ke = np.repeat(K[:1], 50, axis=0)
    out, lse = oracle.decode(q, Ke, V, np.array([0, 50]), np.array([50]), H_KV, scale=scale)
    for hq in range(H_Q):
        h = hq // (H_Q // H_KV)
        np.testing.assert_allclose(out[0, hq], synth.bf16_bits_to_f32(V[:, h]).astype(np.float64).mean(0), atol=1e-12)
        x = scale * qd[hq] @ synth.bf16_bits_to_f32(K[0, h])
        assert lse[0, hq] == pytest.approx(x + math.log(50), abs=1e-12)
    # empty sequence: zero output, lse = -inf
    out, lse = oracle.decode(q, K, V, np.array([0, 0]), np.array([0]), H_KV, scale=scale)
    assert np.all(out == 0) and np.all(np.isneginf(lse))


def test_decode_dominant_key_selects_its_value():
    H_Q, H_KV, d, n = 2, 1, 8, 30
    q = np.full((1, H_Q, d), 0x3F80, np.uint16)                 # q = 1 everywhere
    K = np.zeros((n, H_KV, d), np.uint16)
    K[17] = 0x4220                                              # 40.0: score 320 * scale above the rest
    V = synth.normal_bf16(41, 0, n * d).reshape(n, H_KV, d)
    out, _ = oracle.decode(q, K, V, np.array([0, n]), np.array([n]), H_KV, scale=1.0)
    np.testing.assert_allclose(out[0, 0], synth.bf16_bits_to_f32(V[17, 0]), atol=1e-12)


def test_head_sharing_invariant():
    """MHA, GQA and MQA agree when the K/V heads are duplicated copies of one head."""
    H_Q, d, n = 8, 16, 37
    q = synth.normal_bf16(51, 0, H_Q * d).reshape(1, H_Q, d)
    K1 = synth.normal_bf16(51, 1, n * d).reshape(n, 1, d)
    V1 = synth.normal_bf16(51, 2, n * d).reshape(n, 1, d)
    ref, ref_lse = oracle.decode(q, K1, V1, np.array([0, n]), np.array([n]), 1)
    for H_KV in (2, 4, 8):
        out, lse = oracle.decode(q, np.repeat(K1, H_KV, axis=1), np.repeat(V1, H_KV, axis=1),
                                 np.array([0, n]), np.array([n]), H_KV)
        assert np.array_equal(out, ref) and np.array_equal(lse, ref_lse)


def test_gqa_groups_are_contiguous():
    """Query head hq reads KV head hq // g: with distinct heads, each group's
    output equals an MHA run on that head alone."""
    H_Q, H_KV, d, n = 8, 2, 8, 20
    q = synth.normal_bf16(61, 0, H_Q * d).reshape(1, H_Q, d)
    K = synth.normal_bf16(61, 1, n * H_KV * d).reshape(n, H_KV, d)
    V = synth.normal_bf16(61, 2, n * H_KV * d).reshape(n, H_KV, d)
    out, _ = oracle.decode(q, K, V, np.array([0, n]), np.array([n]), H_KV)
    for hq in range(H_Q):
        one, _ = oracle.decode(q[:, hq:hq + 1], K[:, hq // 4:hq // 4 + 1], V[:, hq // 4:hq // 4 + 1],
                               np.array([0, n]), np.array([n]), 1)
        assert np.array_equal(out[0, hq], one[0, 0])


def test_padding_never_read():
    """Positions past a sequence's length (padding / unfilled slots) do not change the output."""
    H_Q, H_KV, d, n = 4, 2, 8, 13
    q = synth.normal_bf16(71, 0, H_Q * d).reshape(1, H_Q, d)
    K = synth.normal_bf16(71, 1, 32 * H_KV * d).reshape(32, H_KV, d)
    V = synth.normal_bf16(71, 2, 32 * H_KV * d).reshape(32, H_KV, d)
    a = oracle.decode(q, K, V, np.array([0, 32]), np.array([n]), H_KV)
    Kp, Vp = K.copy(), V.copy()
    Kp[n:] = 0x7FC0     # NaN
    Vp[n:] = 0x7F80     # inf
    b = oracle.decode(q, Kp, Vp, np.array([0, 32]), np.array([n]), H_KV)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_prefill_rows_are_decodes():
    """Chunk query i equals a decode at length q_start + i + 1; the last row is
    the decode of the whole sequence."""
    H_Q, H_KV, d, q0, nq = 4, 2, 8, 24, 9
    n = q0 + nq
    K = synth.normal_bf16(81, 1, n * H_KV * d).reshape(n, H_KV, d)
    V = synth.normal_bf16(81, 2, n * H_KV * d).reshape(n, H_KV, d)
    q = synth.normal_bf16(81, 0, nq * H_Q * d).reshape(nq, H_Q, d)
    out, lse = oracle.prefill(q, K, V, q0, H_KV)
    for i in (0, 4, nq - 1):
        o, l = oracle.decode(q[i:i + 1], K, V, np.array([0, n]), np.array([q0 + i + 1]), H_KV)
        assert np.array_equal(out[i], o[0]) and np.array_equal(lse[i], l[0])
    # and against the from-scratch causal computation for the last row
    rng = np.random.default_rng(0)
    ro, rl = _torch_causal_last_row(synth.bf16_bits_to_f32(q[-1]).astype(np.float64),
                                    _dequant(K), _dequant(V), H_Q, float(np.float32(1 / math.sqrt(d))), rng)
    np.testing.assert_allclose(out[-1], ro, atol=1e-12)
    np.testing.assert_allclose(lse[-1], rl, atol=1e-12)


# ---------------------------------------------------------------- int4
def test_int4_codec_nearest_even_and_clamped():
    ys = list(np.arange(-9.0, 9.0, 0.25)) + [0.5, 1.5, 2.5, -0.5, -2.5, 6.5, -6.5, 7.5, -7.5, 1e9, -1e9, 3.4999998]
    ys += list(synth.normal_f64(4, 1, 2000) * 4)
    for y in ys:
        y = float(np.float32(y))
        cand = np.arange(-7, 8)
        dist = np.abs(cand - y)
        best = cand[dist == dist.min()]
        want = int(best[0]) if len(best) == 1 else int(best[best % 2 == 0][0])
        assert oracle.int4_encode(y) == want + 8, y
        assert oracle.int4_encode(y) == int(np.clip(np.rint(np.float32(y)), -7, 7)) + 8     # numpy's rint: ties to even
    assert oracle.int4_encode(float("nan")) == 8
    for q in range(-7, 8):
        assert oracle.int4_decode(q + 8) == q and oracle.int4_encode(float(q)) == q + 8


def test_int4_scales_definition():
    x = synth.normal_bf16(6, 2, 50 * 3 * 8).reshape(50, 3, 8)
    assert np.array_equal(oracle.int4_scales(x), (np.abs(synth.bf16_bits_to_f32(x)).max(axis=0) / np.float32(7)))
    assert np.array_equal(oracle.int4_scales(np.zeros((2, 1, 4), np.uint16)), np.ones((1, 4), np.float32))


def test_int4_pool_image_packs_two_channels_per_byte():
    H, d, bs, N = 2, 8, 4, 6
    img = oracle.PoolImage(N, bs, 1, H, d, "int4", fill=0x00)
    assert img.bytes.size == N * 2 * H * bs * d // 2
    x = synth.normal_bf16(8, 1, 9 * H * d).reshape(9, H, d)
    sc = oracle.int4_scales(x)
    img.scales[0] = np.stack([sc, sc])
    bt = np.array([[3, 0, 5]], np.int32)
    assert img.write_tokens(0, bt, np.array([0], np.int32), np.array([0, 9], np.int64), x, x) == oracle.OK
    st, k, v = img.gather(0, bt[0], 9)
    q = oracle.quantize_int4(x, sc)
    assert st == oracle.OK and np.array_equal(k, q) and np.array_equal(v, q)
    # channel 2j of a row sits in the low nibble of a byte, 2j+1 in the high nibble
    off = img.offset(0, 3, 0, 1, 2, 4)          # block 3, keys, head 1, slot 2, channel 4
    assert off % 2 == 0
    byte = int(img.bytes[off // 2])
    assert byte & 0x0F == q[2, 1, 4] and byte >> 4 == q[2, 1, 5]


def test_decode_equals_full_recompute_int4():
    rng = np.random.default_rng(8)
    H_Q, H_KV, d, lens = 8, 2, 16, [1, 9, 30]
    B = len(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    Kb = synth.normal_bf16(31, 1, int(cu[-1]) * H_KV * d).reshape(-1, H_KV, d)
    Vb = synth.normal_bf16(31, 2, int(cu[-1]) * H_KV * d).reshape(-1, H_KV, d)
    sc = np.stack([oracle.int4_scales(Kb), oracle.int4_scales(Vb)])
    K, V = oracle.quantize_int4(Kb, sc[0]), oracle.quantize_int4(Vb, sc[1])
    q = synth.normal_bf16(32, 1, B * H_Q * d).reshape(B, H_Q, d)
    out, lse = oracle.decode(q, K, V, cu, np.array(lens), H_KV, scales=sc, scale=0.25, kind="int4")
    for b in range(B):
        Kd = (K[cu[b]:cu[b + 1]].astype(np.float64) - 8) * sc[0].astype(np.float64)[None]
        Vd = (V[cu[b]:cu[b + 1]].astype(np.float64) - 8) * sc[1].astype(np.float64)[None]
        ro, rl = _torch_causal_last_row(synth.bf16_bits_to_f32(q[b]).astype(np.float64), Kd, Vd, H_Q, 0.25, rng)
        np.testing.assert_allclose(out[b], ro, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[b], rl, rtol=0, atol=1e-12)
