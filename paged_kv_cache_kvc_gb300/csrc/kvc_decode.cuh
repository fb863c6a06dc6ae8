// Paged decode attention over a block table, split-K with an online softmax.
//
// What it computes ("KV cache: Generation state, latency, and allocation"
// 21.1 and 21.5): for sequence b, KV head h and each of its g query heads,
// softmax(scale * q K^T) V over the n = lens[b] positions that the table maps,
// excluding every slot at or past n.
//
// Work decomposition
//   grid (split, h, b); 128 threads = 4 warps.  A CTA owns logical blocks
//   [split*chunk, min(nblk, (split+1)*chunk)) of (b, h) and all g query heads
//   that share KV head h, so each KV byte leaves HBM once.  Warp w takes the
//   CTA's blocks w, w+4, w+8, ... and keeps its own running max / sum / output.
//   Each warp runs a private ring of R shared-memory stages: one elected lane
//   issues tensor-memory-accelerator (TMA) tile loads of a block's 16 key rows
//   and 16 value rows (one contiguous run in the pool) per 128-byte column band,
//   completing on the stage's mbarrier; the warp waits (bounded), computes, and
//   refills the stage with the block R ahead.
//
// Per 16-token block, on tensor cores (mma.sync m16n8k16, fp32 accumulation):
//   S^T[16 tok x 8q] = K[16 x D] * Q^T[D x 8q]        (tokens are the M dimension,
//                                                      so g <= 8 pads only to N = 8)
//   online softmax over the tokens (warp shuffles across the 8 lanes of a column)
//   O^T[D x 8q]     += V^T[D x 16] * P^T[16 x 8q]     (P^T by movmatrix from S^T)
// bf16 pools feed bf16 operands; P is split into a bf16 high and low part
// (two mma) so the value mixture keeps ~16 bits of each weight.  e4m3 and
// int4 pools convert codes / nibbles to f16 in registers (exact) and fold the
// key scales into q (f16) and the value scales into the output.
//
// TMA writes the tiles with the 128-byte swizzle: within each 128-byte row of
// a band, 16-byte chunk c sits at c ^ (row mod 8), so the ldmatrix and 16-byte
// loads below hit 8 distinct bank groups.
#pragma once
#include <cfloat>
#include <cmath>

#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace kvc {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kBS = 16;                 // positions per block = mma M tile
constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kRescaleSlack = 8.f;   // log2 units: stale reference maxima keep weights <= 256

// stored element kinds of a pool
constexpr int KV_BF16 = 0, KV_E4M3 = 1, KV_INT4 = 2;

template <int D, int KIND>
struct DecodeCfg {
    static constexpr int BITS = KIND == KV_BF16 ? 16 : (KIND == KV_E4M3 ? 8 : 4);
    static constexpr int ROW_BYTES = D * BITS / 8;         // one token row of one head
    static constexpr int STAGE = 2 * kBS * ROW_BYTES;      // keys then values of one (block, head)
    // bf16 / e4m3: the tensor map's rows are token rows and a box is one 128-byte
    // column band of 32 rows; int4 (64-byte rows): rows are 128-byte lines
    // holding two token rows and one box is the whole stage.
    static constexpr bool LINES = ROW_BYTES < 128;
    static constexpr int BANDS = LINES ? 1 : ROW_BYTES / 128;
    static constexpr int BOX_BYTES = LINES ? STAGE : 2 * kBS * 128;
    static constexpr int BOX_ROWS = LINES ? STAGE / 128 : 2 * kBS;
    static constexpr int BOX_X = LINES ? 0 : 128 * 8 / BITS;   // elements per band row
    static constexpr int CHUNKS = ROW_BYTES / 16;             // 16-byte chunks per token row
    // ring bytes per CTA, sized for CTAs per SM (measured on GB300): bf16 64 KiB (2 stages a warp,
    // 3 CTAs an SM), e4m3 48 KiB (3 stages, 4 CTAs), int4 4 stages
    static constexpr int RING_BYTES = KIND == KV_E4M3 ? 49152 : (KIND == KV_BF16 ? 65536 : 98304);
    static constexpr int R0 = RING_BYTES / (kWarps * STAGE);
    static constexpr int R = R0 < 2 ? 2 : (R0 > 4 ? 4 : R0);   // ring depth per warp
    static constexpr int KSTEPS = D / 16;
    static constexpr int MT = D / 16;
    static_assert(LINES ? (ROW_BYTES == 64) : (ROW_BYTES % 128 == 0), "rows: 64 bytes or whole 128-byte bands");
};

// In-kernel split merges hold rows x splits weights plus rows inverse sums in the
// CTA's shared memory, so the host enables them only up to this many partial rows.
constexpr int kMergeRowsMax = 4096;

template <int D, int NT, int KIND>
__host__ __device__ constexpr int decode_smem_bytes()
{
    using C = DecodeCfg<D, KIND>;
    constexpr int stages = kWarps * C::R * C::STAGE;
    constexpr int combine = (kWarps * NT * 8 * 2 + kWarps * NT * 8 * D) * 4;
    constexpr int region = stages > combine ? stages : combine;
    static_assert(region >= (kMergeRowsMax + 32) * 4, "room for the in-kernel merge's weights");
    return 1024 /* alignment slack */ + region + kWarps * C::R * 8 /* mbarriers */;
}

// byte offset of (row, 16-byte chunk) inside a stage, 128-byte swizzle
__device__ __forceinline__ uint32_t swz(int row, int ch)
{
    const int band = ch >> 3, c = ch & 7;
    return static_cast<uint32_t>((band * 2 * kBS + row) * 128 + ((c ^ (row & 7)) << 4));
}

// same for 64-byte token rows packed two per 128-byte line (int4, d_h 128):
// row r is half r & 1 of line r >> 1
__device__ __forceinline__ uint32_t swz64(int row, int ch)
{
    const int line = row >> 1, c = ((row & 1) << 2) + ch;
    return static_cast<uint32_t>(line * 128 + ((c ^ (line & 7)) << 4));
}

template <int D, int KIND>
__device__ __forceinline__ uint32_t row_chunk(int row, int ch)
{
    if constexpr (DecodeCfg<D, KIND>::LINES) return swz64(row, ch);
    else return swz(row, ch);
}

// int4: two nibbles at bits 0..3 and 16..19 of x (stored q + 8) -> f16x2 of q, exact
__device__ __forceinline__ uint32_t nibbles_to_f16x2(uint32_t x)
{
    const uint32_t biased = (x & 0x000F000Fu) | 0x64006400u;      // f16 1024 + u
    uint32_t r;
    asm("sub.f16x2 %0, %1, %2;" : "=r"(r) : "r"(biased), "r"(0x64086408u));   // - (1024 + 8)
    return r;
}

// int4: the nibbles at bits 4..7 and 20..23 of x -> f16x2 of q, exact: masked into
// the mantissa they read 1024 + 16 u, and (1024 + 16 u) / 16 - 72 = u - 8 in one fma
__device__ __forceinline__ uint32_t nibbles_hi_to_f16x2(uint32_t x)
{
    const uint32_t biased = (x & 0x00F000F0u) | 0x64006400u;
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(biased), "r"(0x2C002C00u), "r"(0xD480D480u));
    return r;
}

// int4 quantisation of one value: rint(x / s) clamped to [-7, 7], stored + 8; NaN stores 0
__device__ __forceinline__ uint32_t int4_code(float x, float s)
{
    const float y = __fdiv_rn(x, s);
    if (isnan(y)) return 8u;
    const float r = fminf(fmaxf(rintf(y), -7.f), 7.f);
    return static_cast<uint32_t>(static_cast<int>(r) + 8);
}

// Positions attended by unit b: lens[b] (+1 when the step's token is appended
// in the same launch); for a prefill chunk, whose unit b holds query positions
// b*ppu .. b*ppu+ppu-1 and query i reads len_base + i + 1 positions, the
// longest of its queries.
__device__ __forceinline__ int seq_len(const DecodeParams &p, int b)
{
    if (!p.lens) return p.len_base + min(p.n_pos, (b + 1) * p.ppu);
    return __ldg(p.lens + b) + (p.k_new ? 1 : 0);
}

// Fused append ("KV cache: Generation state, latency, and allocation" Eq. 21.6):
// store sequence b's new key and value rows of head h at (phys, slot) in the
// pool, and put the same stored bytes into the landed stage, so attention uses
// exactly what the pool now holds.  Lanes [0, CH) take the key row, [CH, 2CH)
// the value row, one 16-byte chunk each.
template <int D, int KIND>
__device__ __forceinline__ void append_row(const DecodeParams &p, uint32_t st, int b, int h, int64_t phys, int slot,
                                           int lane)
{
    using C = DecodeCfg<D, KIND>;
    constexpr int CH = C::CHUNKS;
    static_assert(2 * CH <= 32, "one warp covers both rows");
    if (lane >= 2 * CH) return;
    const int kv = lane / CH, ch = lane - kv * CH;
    const uint16_t *src = (kv ? p.v_new : p.k_new) + (static_cast<size_t>(b) * p.H_KV + h) * D;
    uint4 val;
    if constexpr (KIND == KV_BF16) {
        val = *reinterpret_cast<const uint4 *>(src + ch * 8);
    } else if constexpr (KIND == KV_INT4) {   // 32 channels -> 16 bytes, channel 2j in the low nibble
        const float *sc = (kv ? p.s_v : p.s_k) + static_cast<size_t>(h) * D + ch * 32;
        uint32_t o[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int part = 0; part < 4; ++part) {
            const uint4 x = *reinterpret_cast<const uint4 *>(src + ch * 32 + part * 8);
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float f = (i & 1) ? bf16_hi(w[i >> 1]) : bf16_lo(w[i >> 1]);
                o[part] |= int4_code(f, __ldg(sc + part * 8 + i)) << (4 * i);
            }
        }
        val = make_uint4(o[0], o[1], o[2], o[3]);
    } else {
        const uint4 x0 = *reinterpret_cast<const uint4 *>(src + ch * 16);
        const uint4 x1 = *reinterpret_cast<const uint4 *>(src + ch * 16 + 8);
        const uint32_t w[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        const float *sc = (kv ? p.s_v : p.s_k) + static_cast<size_t>(h) * D + ch * 16;
        uint32_t o[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float f = (i & 1) ? bf16_hi(w[i >> 1]) : bf16_lo(w[i >> 1]);
            const uint32_t q = __nv_cvt_float_to_fp8(__fdiv_rn(f, __ldg(sc + i)), __NV_SATFINITE, __NV_E4M3);
            o[i >> 2] |= q << (8 * (i & 3));
        }
        val = make_uint4(o[0], o[1], o[2], o[3]);
    }
    const int64_t e = ((((static_cast<int64_t>(p.layer) * p.N + phys) * p.H_KV + h) * 2 + kv) * kBS + slot) * D;
    *reinterpret_cast<uint4 *>(p.pool + e * C::BITS / 8 + ch * 16) = val;
    sts128(st + row_chunk<D, KIND>(kv * kBS + slot, ch), val);
}

// One 16-token block's update of a warp's running softmax state: scores of the
// block's keys against the warp's query columns, masking (positions at or past
// `valid` in the block; CAUSAL: per column, positions at or past clen), the
// online rescale, and the value mixture.  `st` is the landed stage (keys in
// rows 0..15, values in rows 16..31); tok0 is the block's first position.
template <int D, int NT, int KIND, bool PSPLIT, bool CAUSAL>
__device__ __forceinline__ void block_update(uint32_t st, const uint32_t (&qf)[NT][D / 16][2], float (&m_run)[NT][2],
                                             float (&l_run)[NT][2], float (&oacc)[D / 16][NT][4], int valid, int tok0,
                                             const int (&clen)[NT][2], float scale_log2, int lane)
{
    using C = DecodeCfg<D, KIND>;
    constexpr bool INT4 = KIND == KV_INT4, QUANT = KIND != KV_BF16;
    const int gq = lane >> 2, tg = lane & 3;
    // ---- S^T = K Q^T; with one n-tile, even and odd k-steps accumulate apart (two
    // dependent mma chains of D/32 instead of one of D/16), summed after
    constexpr int NACC = NT == 1 ? 2 : 1;
    float sc[NT][4], sc2[NT][4];
#pragma unroll
    for (int jn = 0; jn < NT; ++jn)
#pragma unroll
        for (int c = 0; c < 4; ++c) sc[jn][c] = sc2[jn][c] = 0.f;
    auto acc = [&](int jn, int kk) -> float(&)[4] { return (NACC == 2 && (kk & 1)) ? sc2[jn] : sc[jn]; };
    if constexpr (!QUANT) {
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
            uint32_t a[4];
            ldsm_x4(a, st + swz((lane & 7) + ((lane >> 3) & 1) * 8, 2 * kk + (lane >> 4)));
#pragma unroll
            for (int jn = 0; jn < NT; ++jn) mma_bf16(acc(jn, kk), a, qf[jn][kk]);
        }
    } else if constexpr (INT4) {
        uint32_t kw[2][4];   // rows gq, gq+8: this thread's 32-channel chunk tg (8 nibbles a word)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const uint4 v = lds128(st + swz64(gq + 8 * r, tg));
            kw[r][0] = v.x;
            kw[r][1] = v.y;
            kw[r][2] = v.z;
            kw[r][3] = v.w;
        }
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
            const int sh = 8 * (kk & 1);   // nibbles (2e, 2e+4) and (2e+1, 2e+5) of word kk / 2
            const uint32_t w0 = kw[0][kk >> 1] >> sh, w1 = kw[1][kk >> 1] >> sh;
            uint32_t a[4];
            a[0] = nibbles_to_f16x2(w0);
            a[2] = nibbles_hi_to_f16x2(w0);
            a[1] = nibbles_to_f16x2(w1);
            a[3] = nibbles_hi_to_f16x2(w1);
#pragma unroll
            for (int jn = 0; jn < NT; ++jn) mma_f16(acc(jn, kk), a, qf[jn][kk]);
        }
    } else {
        uint32_t kw[2][D / 16];   // rows gq, gq+8: this thread's D/4 code bytes each
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int u = 0; u < D / 64; ++u) {
                const uint4 v = lds128(st + swz(gq + 8 * r, (D / 64) * tg + u));
                kw[r][4 * u + 0] = v.x;
                kw[r][4 * u + 1] = v.y;
                kw[r][4 * u + 2] = v.z;
                kw[r][4 * u + 3] = v.w;
            }
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
            uint32_t a[4];
            e4m3x4_to_f16x2x2(kw[0][kk], a[0], a[2]);
            e4m3x4_to_f16x2x2(kw[1][kk], a[1], a[3]);
#pragma unroll
            for (int jn = 0; jn < NT; ++jn) mma_f16(acc(jn, kk), a, qf[jn][kk]);
        }
    }
    if constexpr (NACC == 2)
#pragma unroll
        for (int c = 0; c < 4; ++c) sc[0][c] += sc2[0][c];

    // ---- online softmax (log2 domain); column = query head, rows = tokens gq, gq+8.
    // Decode instances move a column's reference max m_run only when a block's max
    // exceeds it by more than kRescaleSlack (log2 units): below that the weights
    // 2^(s - m_run) stay under 2^kRescaleSlack, l and O keep the same reference, and
    // the output accumulators need no rescale -- the warp skips it unless one of its
    // columns moved (conditional rescaling, as in FlashAttention-4).  The merge and
    // lse use each partial's own reference, so the result is the same softmax.
    uint32_t pb[NT][2], pl[NT][2];
    float alpha[NT][2];
    bool moved = false;
    #pragma unroll
    for (int jn = 0; jn < NT; ++jn) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            if constexpr (CAUSAL) {
                const int tok = tok0 + gq + ((c >> 1) << 3);
                sc[jn][c] = tok < clen[jn][c & 1] ? sc[jn][c] * scale_log2 : -INFINITY;
            } else {   // every column sees the same positions; padding columns hold q = 0
                sc[jn][c] = gq + ((c >> 1) << 3) < valid ? sc[jn][c] * scale_log2 : -INFINITY;
            }
        }
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            float bm = fmaxf(sc[jn][c], sc[jn][c + 2]);
            bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 4));
            bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 8));
            bm = fmaxf(bm, __shfl_xor_sync(kFull, bm, 16));
            float mref;
            if constexpr (CAUSAL) {
                const float mn = fmaxf(m_run[jn][c], bm);
                mref = mn == -INFINITY ? 0.f : mn;   // a column with nothing visible yet
                alpha[jn][c] = fast_exp2(m_run[jn][c] - mref);
                m_run[jn][c] = mn;
                moved = true;
            } else {   // bm is finite: a block has a valid token (the first block always moves)
                const bool up = bm > m_run[jn][c] + kRescaleSlack;
                mref = up ? bm : m_run[jn][c];
                alpha[jn][c] = up ? fast_exp2(m_run[jn][c] - bm) : 1.f;
                m_run[jn][c] = mref;
                moved |= up;
            }
            const float p0 = fast_exp2(sc[jn][c] - mref), p1 = fast_exp2(sc[jn][c + 2] - mref);
            l_run[jn][c] = l_run[jn][c] * alpha[jn][c] + p0 + p1;
            sc[jn][c] = p0;
            sc[jn][c + 2] = p1;
        }
        if constexpr (!QUANT) {
            const uint32_t h0 = pack_bf16(sc[jn][0], sc[jn][1]), h1 = pack_bf16(sc[jn][2], sc[jn][3]);
            pb[jn][0] = movmatrix_trans(h0);
            pb[jn][1] = movmatrix_trans(h1);
            if constexpr (PSPLIT) {
                pl[jn][0] = movmatrix_trans(pack_bf16(sc[jn][0] - bf16_lo(h0), sc[jn][1] - bf16_hi(h0)));
                pl[jn][1] = movmatrix_trans(pack_bf16(sc[jn][2] - bf16_lo(h1), sc[jn][3] - bf16_hi(h1)));
            }
        } else {
            pb[jn][0] = movmatrix_trans(pack_f16(sc[jn][0], sc[jn][1]));
            pb[jn][1] = movmatrix_trans(pack_f16(sc[jn][2], sc[jn][3]));
        }
    }
    if (CAUSAL || __any_sync(kFull, moved)) {
#pragma unroll
        for (int jn = 0; jn < NT; ++jn)
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    oacc[mt][jn][c] *= alpha[jn][c];
                    oacc[mt][jn][c + 2] *= alpha[jn][c];
                }
    }

    // ---- O^T += V^T P^T
    if constexpr (!QUANT) {
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
            uint32_t a[4];
            ldsm_x4_trans(a, st + swz(kBS + (lane & 7) + ((lane >> 4) & 1) * 8, 2 * mt + ((lane >> 3) & 1)));
#pragma unroll
            for (int jn = 0; jn < NT; ++jn) {
                mma_bf16(oacc[mt][jn], a, pb[jn]);
                if constexpr (PSPLIT) mma_bf16(oacc[mt][jn], a, pl[jn]);
            }
        }
    } else if constexpr (INT4) {
        // output channels permuted as for e4m3: m-row gq of tile mt is channel 16*gq + 2*mt,
        // m-row gq+8 the next one; the thread's 16 channels are 8 bytes of each value row
        // value rows 2tg, 2tg+1, 2tg+8, 2tg+9.  Lanes with odd tg load each pair in the other
        // order, so that every load's four lines (two token rows each) use all eight 16-byte
        // chunk slots of the 128-byte swizzle (two wavefronts, not four); the byte
        // selectors below put the pair back in order.
        const uint32_t par = static_cast<uint32_t>(tg & 1);
        uint32_t vw[4][2];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int row = kBS + 2 * tg + ((r & 1) ^ static_cast<int>(par)) + (r >> 1) * 8;
            const uint32_t a = st + swz64(row, gq >> 1) + 8 * (gq & 1);
            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(vw[r][0]), "=r"(vw[r][1]) : "r"(a));
        }
        // selector of byte k: [row 2tg .b_k, same, row 2tg+1 .b_k, same]
        const uint32_t sel0 = par ? 0x0044u : 0x4400u;
#pragma unroll
        for (int w = 0; w < 2; ++w)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t sel = sel0 + 0x1111u * static_cast<uint32_t>(k);
                const uint32_t x01 = __byte_perm(vw[0][w], vw[1][w], sel);
                const uint32_t x89 = __byte_perm(vw[2][w], vw[3][w], sel);
                const uint32_t a[4] = {nibbles_to_f16x2(x01), nibbles_hi_to_f16x2(x01),
                                       nibbles_to_f16x2(x89), nibbles_hi_to_f16x2(x89)};
#pragma unroll
                for (int jn = 0; jn < NT; ++jn) mma_f16(oacc[4 * w + k][jn], a, pb[jn]);
            }
    } else {
        // output channels permuted: m-row r of tile mt is channel gq*D/8 + 2*mt (+1 for r >= 8)
        uint32_t vw[4][D / 32];   // value rows 2tg, 2tg+1, 2tg+8, 2tg+9; D/8 code bytes each
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int u = 0; u < D / 128; ++u) {
                const uint4 v = lds128(st + swz(kBS + 2 * tg + (r & 1) + (r >> 1) * 8, (D / 128) * gq + u));
                vw[r][4 * u + 0] = v.x;
                vw[r][4 * u + 1] = v.y;
                vw[r][4 * u + 2] = v.z;
                vw[r][4 * u + 3] = v.w;
            }
#pragma unroll
        for (int w = 0; w < D / 32; ++w) {
            const uint32_t x01 = __byte_perm(vw[0][w], vw[1][w], 0x5140);
            const uint32_t y01 = __byte_perm(vw[0][w], vw[1][w], 0x7362);
            const uint32_t x89 = __byte_perm(vw[2][w], vw[3][w], 0x5140);
            const uint32_t y89 = __byte_perm(vw[2][w], vw[3][w], 0x7362);
            uint32_t a0[4], a1[4];
            e4m3x4_to_f16x2x2(x01, a0[0], a0[1]);
            e4m3x4_to_f16x2x2(x89, a0[2], a0[3]);
            e4m3x4_to_f16x2x2(y01, a1[0], a1[1]);
            e4m3x4_to_f16x2x2(y89, a1[2], a1[3]);
#pragma unroll
            for (int jn = 0; jn < NT; ++jn) {
                mma_f16(oacc[2 * w][jn], a0, pb[jn]);
                mma_f16(oacc[2 * w + 1][jn], a1, pb[jn]);
            }
        }
    }
}

// CAUSAL: columns may see different numbers of positions (prefill tiles), so
// the mask is per column and a column may see nothing in a block; decode
// instances (every column sees the unit's whole length) skip both.
// One CTA of the split kernel: split `split` of unit (b, h).
template <int D, int NT, int KIND, bool PSPLIT, bool CAUSAL>
__device__ __forceinline__ void decode_cta(const CUtensorMap &tmap, const DecodeParams &p, const int split,
                                           const int h, const int b)
{
    using C = DecodeCfg<D, KIND>;
    constexpr bool INT4 = KIND == KV_INT4, QUANT = KIND != KV_BF16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tg = lane & 3;
    const int hq0 = h * p.g;
    // query columns of the unit: ppu consecutive positions x the g heads of KV head h
    // (decode instances have one position per unit: no divisions)
    const int rows = CAUSAL ? p.ppu * p.g : p.g;
    auto col_pos = [&](int qi) { return CAUSAL ? b * p.ppu + qi / p.g : b; };
    auto col_real = [&](int qi) { return CAUSAL ? (qi < rows && col_pos(qi) < p.n_pos) : qi < rows; };
    auto col_orow = [&](int qi) {   // row of the column in q / out ([position][H_Q])
        return CAUSAL ? static_cast<size_t>(col_pos(qi)) * p.H_Q + hq0 + qi % p.g
                      : static_cast<size_t>(b) * p.H_Q + hq0 + qi;
    };

    int len = seq_len(p, b);
    if (len < 0 || static_cast<int64_t>(len) > static_cast<int64_t>(p.max_blocks) * kBS) {
        if (split == 0 && threadIdx.x == 0) atomicOr(p.err, KVC_EBIT_RANGE);
        len = 0;
    }
    const int nblk = (len + kBS - 1) / kBS;
    if (nblk == 0) {   // empty sequence: zero output, lse = -inf
        if (split == 0) {
            for (int i = threadIdx.x; i < rows * D; i += kThreads)
                if (col_real(i / D)) p.out[col_orow(i / D) * D + i % D] = 0.f;
            if (p.lse && threadIdx.x < rows && col_real(threadIdx.x)) p.lse[col_orow(threadIdx.x)] = -INFINITY;
        }
        return;
    }
    const int blk0 = split * p.chunk;
    if (blk0 >= nblk) return;
    const int nloc = min(nblk, blk0 + p.chunk) - blk0;
    const int32_t *bt_row = p.bt + static_cast<int64_t>(b) * p.bt_stride + blk0 + warp;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (decode_smem_bytes<D, NT, KIND>() - 1024 - kWarps * C::R * 8));
    if (lane == 0) {
        for (int s = 0; s < C::R; ++s) mbar_init(smem_u32(&bars[warp * C::R + s]), 1);
        fence_barrier_init();
    }
    if (threadIdx.x == 0) prefetch_tensormap(&tmap);
    __syncthreads();

    const int nmine = nloc > warp ? (nloc - warp + kWarps - 1) / kWarps : 0;   // this warp's blocks
    const uint32_t st_base = smem_u32(smem + warp * C::R * C::STAGE);
    const uint32_t bar_base = smem_u32(&bars[warp * C::R]);
    const int64_t row_layer = static_cast<int64_t>(p.layer) * p.N;

    // Table entries of this warp's blocks, 32 at a time in registers: lane i
    // holds local block 32*k + i of the current batch (t_cur) and the next (t_next).
    auto load_entry = [&](int jj) -> int32_t { return jj < nmine ? __ldg(bt_row + kWarps * jj) : -1; };
    int32_t t_cur = load_entry(lane), t_next = load_entry(32 + lane);
    auto entry = [&](int jj, int jbase) -> int32_t {
        const int32_t v = (jj - jbase < 32) ? t_cur : t_next;
        return __shfl_sync(kFull, v, (jj - jbase) & 31);
    };
    auto issue = [&](int jj, int jbase) {   // warp-collective; lane 0 issues
        const int32_t phys = entry(jj, jbase);
        if (lane == 0 && !p.stall_loads) {
            const uint32_t bar = bar_base + 8u * static_cast<uint32_t>(jj % C::R);
            if (phys < 0 || static_cast<int64_t>(phys) >= p.N) {
                atomicOr(p.err, KVC_EBIT_BAD_BLOCK);
                mbar_arrive(bar);   // complete the phase without data; the consumer skips it
            } else {
                const int32_t y = static_cast<int32_t>(((row_layer + phys) * p.H_KV + h) * C::BOX_ROWS);
                const uint32_t dst = st_base + static_cast<uint32_t>((jj % C::R) * C::STAGE);
                mbar_arrive_expect_tx(bar, C::STAGE);
#pragma unroll
                for (int band = 0; band < C::BANDS; ++band)
                    tma_load_2d(dst + band * C::BOX_BYTES, &tmap, bar, band * C::BOX_X, y);
            }
        }
    };

    // ---- query fragments (B operand, k = channel, n = query head of the group)
    uint32_t qf[NT][C::KSTEPS][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int qi = 8 * j + gq;
        const bool real = col_real(qi);
        const uint16_t *qrow = p.q + (real ? col_orow(qi) : static_cast<size_t>(0)) * D;
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
            if constexpr (!QUANT) {
                qf[j][kk][0] = real ? *reinterpret_cast<const uint32_t *>(qrow + 16 * kk + 2 * tg) : 0u;
                qf[j][kk][1] = real ? *reinterpret_cast<const uint32_t *>(qrow + 16 * kk + 8 + 2 * tg) : 0u;
            } else if constexpr (INT4) {
                // slots of k-step kk: channels base, base+4 (b0) and base+1, base+5 (b1) of the
                // thread's 32-channel chunk, matching the nibble pairs the key fragments hold
                const int base = 32 * tg + 8 * (kk >> 1) + 2 * (kk & 1);
                const float *sk = p.s_k + static_cast<size_t>(h) * D;
                auto qv = [&](int c) {
                    const uint16_t raw = real ? qrow[c] : uint16_t(0);
                    return __uint_as_float(static_cast<uint32_t>(raw) << 16) * __ldg(sk + c);
                };
                qf[j][kk][0] = pack_f16(qv(base), qv(base + 4));
                qf[j][kk][1] = pack_f16(qv(base + 1), qv(base + 5));
            } else {
                // channel slots permuted: thread tg owns channels [tg*D/4, (tg+1)*D/4), four per k-step
                const int c0 = (D / 4) * tg + 4 * kk;
                const uint2 raw = real ? *reinterpret_cast<const uint2 *>(qrow + c0) : make_uint2(0u, 0u);
                const float *sk = p.s_k + static_cast<size_t>(h) * D + c0;
                qf[j][kk][0] = pack_f16(bf16_lo(raw.x) * __ldg(sk + 0), bf16_hi(raw.x) * __ldg(sk + 1));
                qf[j][kk][1] = pack_f16(bf16_lo(raw.y) * __ldg(sk + 2), bf16_hi(raw.y) * __ldg(sk + 3));
            }
        }
    }

    // positions each of this thread's two columns per n-tile may read (0 for padding columns)
    int clen[NT][2];
#pragma unroll
    for (int jn = 0; jn < NT; ++jn)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const int qi = 8 * jn + 2 * tg + c;
            clen[jn][c] = !CAUSAL ? len : (!col_real(qi) ? 0 : p.len_base + col_pos(qi) + 1);
        }

    float m_run[NT][2], l_run[NT][2];
    float oacc[C::MT][NT][4];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        m_run[j][0] = m_run[j][1] = -INFINITY;
        l_run[j][0] = l_run[j][1] = 0.f;
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) oacc[mt][j][0] = oacc[mt][j][1] = oacc[mt][j][2] = oacc[mt][j][3] = 0.f;
    }

    for (int jj = 0; jj < min(C::R, nmine); ++jj) issue(jj, 0);

    int j = 0;
    bool timed_out = false;
    for (; j < nmine; ++j) {
        const int jbase = j & ~31;
        if (j > 0 && (j & 31) == 0) {
            t_cur = t_next;
            t_next = load_entry(j + 32 + lane);
        }
        const int s = j % C::R;
        const bool ok = mbar_wait_bounded(bar_base + 8u * s, static_cast<uint32_t>((j / C::R) & 1));
        if (!__all_sync(kFull, ok)) {
            timed_out = true;
            break;
        }
        const int32_t phys = entry(j, jbase);
        if (phys >= 0 && static_cast<int64_t>(phys) < p.N) {
            const uint32_t st = st_base + static_cast<uint32_t>(s * C::STAGE);
            const int valid = min(kBS, len - (blk0 + warp + kWarps * j) * kBS);

            // value rows past the sequence end may hold anything (NaN included): zero them
            // (every int4 nibble is a finite value, and its weight there is 0)
            if (!INT4 && valid < kBS) {
                const int nz = (kBS - valid) * C::BANDS * 8;
                for (int i = lane; i < nz; i += 32) sts128_zero(st + swz(kBS + valid + i / (C::BANDS * 8), i % (C::BANDS * 8)));
            }
            // the step's own token (fused append) is the last valid slot of the last block
            if (p.k_new && blk0 + warp + kWarps * j == nblk - 1) append_row<D, KIND>(p, st, b, h, phys, valid - 1, lane);
            __syncwarp();

            block_update<D, NT, KIND, PSPLIT, CAUSAL>(st, qf, m_run, l_run, oacc, valid,
                                                      (blk0 + warp + kWarps * j) * kBS, clen, p.scale_log2, lane);
        }
        __syncwarp();
        if (j + C::R < nmine) {
            if (lane == 0) fence_proxy_async_smem();
            issue(j + C::R, jbase);
        }
    }

    if (timed_out) {   // record, then let copies already in flight land before the CTA exits
        if (lane == 0) {
            atomicOr(p.err, KVC_EBIT_TIMEOUT);
            for (int jj = j; jj < min(nmine, j + C::R); ++jj)
                (void)mbar_wait_bounded(bar_base + 8u * (jj % C::R), static_cast<uint32_t>((jj / C::R) & 1), 100000000ull);
        }
        __syncwarp();
    }

#pragma unroll
    for (int jn = 0; jn < NT; ++jn)
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            float l = l_run[jn][c];
            l += __shfl_xor_sync(kFull, l, 4);
            l += __shfl_xor_sync(kFull, l, 8);
            l += __shfl_xor_sync(kFull, l, 16);
            l_run[jn][c] = l;
        }

    // ---- combine the four warps (shared memory reused), then write
    __syncthreads();
    constexpr int QW = NT * 8;
    float *cm = reinterpret_cast<float *>(smem);
    float *cl = cm + kWarps * QW;
    float *co = cl + kWarps * QW;
#pragma unroll
    for (int jn = 0; jn < NT; ++jn) {
#pragma unroll
        for (int c = 0; c < 2; ++c)
            if (gq == 0) {
                cm[warp * QW + 8 * jn + 2 * tg + c] = m_run[jn][c];
                cl[warp * QW + 8 * jn + 2 * tg + c] = l_run[jn][c];
            }
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int qi = 8 * jn + 2 * tg + (c & 1);
                const int dim = QUANT ? gq * (D / 8) + 2 * mt + (c >> 1) : 16 * mt + gq + 8 * (c >> 1);
                co[(warp * QW + qi) * D + dim] = oacc[mt][jn][c];
            }
    }
    __syncthreads();

    const int ns = (nblk + p.chunk - 1) / p.chunk;
    for (int i = threadIdx.x; i < rows * D; i += kThreads) {
        const int qi = i / D, d = i - qi * D;
        if (!col_real(qi)) continue;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, cm[w * QW + qi]);
        const float Mref = M == -INFINITY ? 0.f : M;     // no visible position in this CTA's blocks
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float e = fast_exp2(cm[w * QW + qi] - Mref);   // warps without blocks: exp2(-inf) = 0
            L += e * cl[w * QW + qi];
            O += e * co[(w * QW + qi) * D + d];
        }
        if constexpr (QUANT) O *= __ldg(p.s_v + static_cast<size_t>(h) * D + d);
        const size_t bq = col_orow(qi);
        if (ns == 1) {
            p.out[bq * D + d] = O / L;
            if (d == 0 && p.lse) p.lse[bq] = (M + log2f(L)) * kLn2;
        } else {
            const size_t pi = bq * p.max_splits + split;
            p.part_o[pi * D + d] = O;
            if (d == 0) p.part_ml[pi] = make_float2(M, L);
        }
    }
    if (ns == 1 || !p.counters) return;   // without counters the host launches the merge kernel

    // ---- split-K merge by the last split CTA of (b, h) to finish: the partial
    // writes above are released by the fence before the count, and acquired
    // by the fence after the last CTA sees ns - 1 earlier arrivals.
    __shared__ uint32_t last_flag;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const uint32_t prev = atomicAdd(p.counters + static_cast<size_t>(b) * p.H_KV + h, 1u);
        last_flag = (prev == static_cast<uint32_t>(ns - 1)) ? 1u : 0u;
    }
    __syncthreads();
    if (!last_flag) return;
    __threadfence();
    // The merge sits at the end of the launch, so it is written for latency: one
    // warp per query column reduces (m, l) over the splits with its lanes and
    // leaves the weights 2^(m_s - M) and 1/L in shared memory (free again: every
    // thread is past the combine); then each thread issues the loads of all of
    // its float4 column's partials at once.  rows * ns <= kMergeRowsMax (host).
    float *wsm = reinterpret_cast<float *>(smem);   // [rows][ns] weights, then [rows] 1/L
    float *linv = wsm + rows * ns;
    for (int qi = warp; qi < rows; qi += kWarps) {
        if (!col_real(qi)) continue;   // warp-uniform
        const size_t bq = col_orow(qi);
        const float2 *ml = p.part_ml + bq * p.max_splits;
        const float2 v0 = lane < ns ? __ldcg(ml + lane) : make_float2(-INFINITY, 0.f);
        float m = v0.x;
        for (int sp = lane + 32; sp < ns; sp += 32) m = fmaxf(m, __ldcg(&ml[sp].x));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
        const float Mref = m == -INFINITY ? 0.f : m;
        float l = 0.f;
        if (lane < ns) {
            const float e = fast_exp2(v0.x - Mref);
            wsm[qi * ns + lane] = e;
            l = e * v0.y;
        }
        for (int sp = lane + 32; sp < ns; sp += 32) {
            const float2 v = __ldcg(ml + sp);
            const float e = fast_exp2(v.x - Mref);
            wsm[qi * ns + sp] = e;
            l += e * v.y;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(kFull, l, o);
        if (lane == 0) {
            linv[qi] = 1.f / l;
            if (p.lse) p.lse[bq] = (m + log2f(l)) * kLn2;
        }
    }
    __syncthreads();
    constexpr int D4 = D / 4;
    for (int i = threadIdx.x; i < rows * D4; i += kThreads) {
        const int qi = i / D4, d4 = i - qi * D4;
        if (!col_real(qi)) continue;
        const size_t bq = col_orow(qi);
        const float4 *po = reinterpret_cast<const float4 *>(p.part_o + bq * p.max_splits * D) + d4;
        const float *w = wsm + qi * ns;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int sp = 0; sp < ns; ++sp) {
            const float4 o = __ldcg(po + static_cast<size_t>(sp) * D4);
            const float e = w[sp];
            acc.x = fmaf(e, o.x, acc.x);
            acc.y = fmaf(e, o.y, acc.y);
            acc.z = fmaf(e, o.z, acc.z);
            acc.w = fmaf(e, o.w, acc.w);
        }
        const float inv = linv[qi];
        reinterpret_cast<float4 *>(p.out + bq * D)[d4] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
    if (threadIdx.x == 0) p.counters[static_cast<size_t>(b) * p.H_KV + h] = 0u;   // ready for the next launch
}

// Lets a programmatic dependent (the split merge) be scheduled once every CTA
// of this grid has started; the dependent waits for this grid's completion
// before it reads anything the grid wrote.
__device__ __forceinline__ void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;"); }

// Holds the CTA until the grid it programmatically depends on (the kernel before it
// on the stream, when launched with programmatic stream serialization) has finished
// and its memory writes are visible; returns at once in an ordinary launch.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// grid (split, KV head, unit)
template <int D, int NT, int KIND, bool PSPLIT, bool CAUSAL>
__global__ void __launch_bounds__(kThreads) decode_kernel(const __grid_constant__ CUtensorMap tmap,
                                                          const DecodeParams p)
{
    using C = DecodeCfg<D, KIND>;
    allow_dependent_launch();
    // While the kernel before it drains: a speculative L2 prefetch of the blocks the CTA's
    // rings load first, from the lengths and table as they stand now (they may still change;
    // nothing here is used but as a cache hint, and the CTA reads them again after the wait).
    if (!CAUSAL && p.lens && p.pool && threadIdx.x < kWarps * C::R) {
        const int b = blockIdx.z, h = blockIdx.y;
        const int len_s = p.lens[b] + (p.k_new ? 1 : 0);
        const int blk = blockIdx.x * p.chunk + threadIdx.x;
        if (blk < p.max_blocks && blk * kBS < len_s) {
            const int32_t e = p.bt[static_cast<int64_t>(b) * p.bt_stride + blk];
            if (e >= 0 && static_cast<int64_t>(e) < p.N)
                prefetch_l2_bulk(p.pool + ((static_cast<int64_t>(p.layer) * p.N + e) * p.H_KV + h) * C::STAGE,
                                 C::STAGE);
        }
    }
    grid_dependency_wait();   // launched as a programmatic dependent: nothing global is touched before this
    decode_cta<D, NT, KIND, PSPLIT, CAUSAL>(tmap, p, blockIdx.x, blockIdx.y, blockIdx.z);
}

// Fetch (and on first use configure) the kernel instance for a shape.
struct DecodeKernel {
    const void *fn;
    int smem;
    int ctas_per_sm;
    int threads = kThreads;   // block size
    bool tmap16 = false;      // takes the pool's 16-row tensor map (else the map of whole blocks)
    int split_unit = 1;       // tensor-memory kernels: blocks per split a multiple of this
};

template <int D, int NT, int KIND, bool PSPLIT, bool CAUSAL = false>
DecodeKernel decode_instance()
{
    static DecodeKernel k = [] {
        DecodeKernel r;
        r.fn = reinterpret_cast<const void *>(&decode_kernel<D, NT, KIND, PSPLIT, CAUSAL>);
        r.smem = decode_smem_bytes<D, NT, KIND>();
        r.ctas_per_sm = 0;
        if (cudaFuncSetAttribute(&decode_kernel<D, NT, KIND, PSPLIT, CAUSAL>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, r.smem) == cudaSuccess) {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, &decode_kernel<D, NT, KIND, PSPLIT, CAUSAL>,
                                                              kThreads, r.smem) == cudaSuccess)
                r.ctas_per_sm = n;
        }
        return r;
    }();
    return k;
}

kvc_status run_decode(const kvc_pool *pool, DecodeParams &p, const DecodeKernel &k, cudaStream_t stream);

// Kernel instance selection without launching (used by the allocation-free entry point).
DecodeKernel select_decode_bf16(int D, int g);
DecodeKernel select_decode_fp8(int D, int g);
DecodeKernel select_decode_int4(int D, int g);
kvc_status launch_split_merge(const DecodeParams &p, int D, cudaStream_t stream);

}  // namespace kvc
