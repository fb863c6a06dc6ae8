// Causal attention of a prefill chunk on the fifth-generation tensor cores,
// queries on the MMA's M dimension, scores and outputs in tensor memory (TMEM)
// ("KV cache: Generation state, latency, and allocation" 21.3: a chunked
// prefill attends over the earlier positions and its own; the xf_kv_cache
// page, "End-to-end flow": the new tokens attend to the shared prefix through
// the row's block table).
//
// Query i of the chunk sits at position q_start + i and reads positions
// 0 .. q_start + i.  A CTA takes KV head h and 128 query rows: 128 / g
// consecutive chunk positions x the g query heads of h (row r = position
// r / g, head h * g + r mod g), so every staged key / value tile serves all g
// heads.  224 threads in three roles:
//   warps 4, 6  TMA producers, warp 4 the key rows and warp 6 the value rows
//               of a stage: 64 keys per stage (4 blocks of the row), each
//               block's rows a 16-row box per 128-byte band (128-byte
//               swizzle), a ring of 5 stages.  Two warps because one warp's
//               boxes are issued one after the other (about 40 ns each).
//   warp 5      MMA issuer (one elected lane), per stage j:
//                 S[128 x 64]  = Q[128 x D] . K^T        (K-major A and B)
//                 O[128 x D]  += P[128 x 64] . V[64 x D]  (K-major A, MN-major B)
//               S and P double-buffered (S in TMEM, P in shared memory), so
//               the scores of stage j + 1 are computed while the softmax of
//               stage j runs, and the softmax of stage j + 1 writes its
//               weights while the value MMA of stage j reads the other buffer.
//   warps 0..3  softmax, thread r = row r (TMEM lane r): the causal mask
//               (key < q_start + position + 1), the row's running maximum as a
//               reference that moves only when a score exceeds it by more than
//               8 (log2 units), then the row's O in TMEM and its sum are
//               rescaled (the warp does it together when any lane needs it,
//               after the value MMA of the stage before has landed in O);
//               P row r as bf16 into shared memory.
// Value rows of positions past the row's end are zeroed before the value MMA
// (a zero weight times NaN is NaN).  The epilogue divides each row by its sum.
#pragma once
#include "kvc_decode_tc.cuh"

namespace kvc {

constexpr int kPtKeys = 64;                     // keys per stage
constexpr int kPtRing = 5;
constexpr int kPtThreads = 224;

template <int D>
struct PrefillTcCfg {
    static constexpr int BANDS = D / 64;                      // 128-byte column bands of a bf16 row
    static constexpr int KBAND = kPtKeys * 128;               // one band of the stage's 64 key rows
    static constexpr int STAGE = 2 * BANDS * KBAND;           // keys, then values
    static constexpr int QBAND = 128 * 128;                   // one band of the 128 query rows
    static constexpr int Q = kPtRing * STAGE;
    static constexpr int P = Q + BANDS * QBAND;               // P[2]: 128 rows x 64 keys bf16 (one band) each
    static constexpr int BARS = P + 2 * 128 * 128;
    static constexpr int NUM_BARS = 2 * kPtRing + 8;          // full, kvfree, s_full[2], s_free[2], p_full[2], pv_done[2]
    static constexpr int SLOT = BARS + NUM_BARS * 8;
    static constexpr int SMEM = 1024 + SLOT + 16;
    static constexpr uint32_t COLS = 256;                     // S[0] 0..63, S[1] 64..127, O from column 128
};

template <int D>
__device__ __forceinline__ void prefill_tc_cta(const CUtensorMap &tmap16, const DecodeParams &p, const int tile,
                                               const int h)
{
    using C = PrefillTcCfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = p.g, ppt = 128 / g;                 // positions per tile
    const int q_start = p.len_base, n_q = p.n_pos;
    const int total = q_start + n_q;                  // positions the row holds
    const int pos0 = tile * ppt;                      // first chunk position of the tile
    const int n_keys = min(total, q_start + pos0 + ppt);
    const int nt = (n_keys + kPtKeys - 1) / kPtKeys;
    const int nblk = (n_keys + kBS - 1) / kBS;
    const int64_t row_layer = static_cast<int64_t>(p.layer) * p.N;

    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + C::BARS;
    auto full_bar = [&](int s) { return bars + 8u * s; };
    auto kvfree_bar = [&](int s) { return bars + 8u * (kPtRing + s); };
    auto sfull_bar = [&](int sb) { return bars + 8u * (2 * kPtRing + sb); };
    auto sfree_bar = [&](int sb) { return bars + 8u * (2 * kPtRing + 2 + sb); };
    auto pfull_bar = [&](int pb) { return bars + 8u * (2 * kPtRing + 4 + pb); };
    auto pvdone_bar = [&](int pb) { return bars + 8u * (2 * kPtRing + 6 + pb); };
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::SLOT);

    if (tid == 0) {
        for (int s = 0; s < kPtRing; ++s) {
            mbar_init(full_bar(s), 2);   // the key producer and the value producer
            mbar_init(kvfree_bar(s), 1);
        }
        for (int sb = 0; sb < 2; ++sb) {
            mbar_init(sfull_bar(sb), 1);
            mbar_init(sfree_bar(sb), 128);
            mbar_init(pfull_bar(sb), 128);
            mbar_init(pvdone_bar(sb), 1);
        }
        fence_barrier_init();
        prefetch_tensormap(&tmap16);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), C::COLS);
        tmem_relinquish();
    }
    if (tid < 128) {   // query row tid (zero past the chunk): the K-major A operand of the score MMA
        const int pos = pos0 + tid / g;
        const uint16_t *qrow = p.q + (static_cast<size_t>(min(pos, n_q - 1)) * p.H_Q + h * g + tid % g) * D;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            const uint4 v = pos < n_q ? *reinterpret_cast<const uint4 *>(qrow + c * 8) : make_uint4(0u, 0u, 0u, 0u);
            sts128(sbase + C::Q + (c >> 3) * C::QBAND + sw128(tid, c & 7), v);
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tm_o = tmem + 128;

    // the row's table entries, 32 (8 stages) at a time in registers, one window ahead: lane l
    // holds block 32 w + l of window w
    constexpr int BPS = kPtKeys / kBS;                // blocks per stage
    auto load_entry = [&](int blk) -> int32_t { return blk < nblk ? __ldg(p.bt + blk) : -1; };

    bool timed_out = false;
    if (warp == 4 || warp == 6) {
        // ------------------------------------------------------------ TMA producers (4: keys, 6: values)
        const int kvp = warp == 6 ? 1 : 0;
        int32_t ecur = load_entry(lane), enext = load_entry(32 + lane);
        int j = 0;
        for (; j < nt; ++j) {
            if (j > 0 && (j % (32 / BPS)) == 0) {
                ecur = enext;
                enext = load_entry((j / (32 / BPS) + 1) * 32 + lane);
            }
            const int s = j % kPtRing;
            if (j >= kPtRing) {
                const bool ok = mbar_wait_bounded(kvfree_bar(s), static_cast<uint32_t>(((j / kPtRing) - 1) & 1));
                if (!__all_sync(kFull, ok)) {
                    timed_out = true;
                    break;
                }
            }
            const int blk = j * BPS + lane;
            const int32_t e = __shfl_sync(kFull, ecur, (j % (32 / BPS)) * BPS + (lane & (BPS - 1)));
            const bool v = lane < BPS && blk < nblk && e >= 0 && static_cast<int64_t>(e) < p.N;
            if (kvp == 0 && lane < BPS && blk < nblk && !v) atomicOr(p.err, KVC_EBIT_BAD_BLOCK);
            const uint32_t mask = __ballot_sync(kFull, v);
            if (lane == 0) {
                if (mask == 0u) mbar_arrive(full_bar(s));
                else mbar_arrive_expect_tx(full_bar(s), static_cast<uint32_t>(__popc(mask)) * C::BANDS * (kBS * 128u));
            }
            __syncwarp();
            // one box per lane, all in one instruction: lane = (band, block); every lane
            // already holds the entry of block lane mod BPS
            const int bl = lane % BPS, band = lane / BPS;
            if (lane < BPS * C::BANDS && ((mask >> bl) & 1u)) {
                const int32_t y = static_cast<int32_t>(((row_layer + e) * p.H_KV + h) * (2 * kBS)) + kvp * kBS;
                tma_load_2d(sbase + s * C::STAGE + (kvp * C::BANDS + band) * C::KBAND + bl * (kBS * 128), &tmap16,
                            full_bar(s), band * 64, y);
            }
        }
        if (lane == 0)
            for (int jj = max(0, j - kPtRing); jj < j; ++jj) {
                (void)mbar_wait_bounded(full_bar(jj % kPtRing), static_cast<uint32_t>((jj / kPtRing) & 1), 100000000ull);
                (void)mbar_wait_bounded(kvfree_bar(jj % kPtRing), static_cast<uint32_t>((jj / kPtRing) & 1),
                                        100000000ull);
            }
        __syncwarp();
    } else if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc_qk = tc_idesc_f16(128, kPtKeys, true, false, false);
        constexpr uint32_t idesc_pv = tc_idesc_f16(128, D, true, false, true);
        // Issues whichever MMA is ready: the value MMA of stage jp once its weights are in
        // shared memory (it releases the stage and the weight buffer), the score MMA of stage
        // jq once its keys have landed and its score buffer is free.  Barriers are tested
        // without blocking.
        int32_t ecur = load_entry(lane), enext = load_entry(32 + lane);
        auto ready = [&](uint32_t bar, uint32_t parity) {   // lane 0 tests, the warp agrees
            const uint32_t r = lane == 0 ? (mbar_test_wait(bar, parity) ? 1u : 0u) : 0u;
            return __shfl_sync(kFull, r, 0) != 0u;
        };
        const uint64_t desc_q = tc_smem_desc(sbase + C::Q, 16, 1024, kSwizzle128B);
        const uint64_t desc_p0 = tc_smem_desc(sbase + C::P, 16, 1024, kSwizzle128B);
        int jq = 0, jp = 0;
        uint64_t idle_since = 0;
        uint32_t idle = 0;
        while (jp < nt) {
            bool progressed = false;
            if (jp < jq && ready(pfull_bar(jp & 1), static_cast<uint32_t>((jp >> 1) & 1))) {
                tc_fence_after();
                {
                    const uint64_t desc_p = tc_desc_advance(desc_p0, (jp & 1) * (128 * 128));
                    const uint64_t b0 = tc_smem_desc(sbase + (jp % kPtRing) * C::STAGE + C::BANDS * C::KBAND, C::KBAND,
                                                     1024, kSwizzle128B);
#pragma unroll
                    for (int kk = 0; kk < kPtKeys / 16; ++kk)   // 16 keys: 32 bytes of P rows, 2048 of V rows
                        tc_mma_f16_warp(tm_o, tc_desc_advance(desc_p, kk * 32), tc_desc_advance(b0, kk * 2048),
                                        idesc_pv, (jp > 0 || kk > 0) ? 1u : 0u);
                    tc_commit_warp(kvfree_bar(jp % kPtRing));
                    tc_commit_warp(pvdone_bar(jp & 1));
                }
                __syncwarp();
                ++jp;
                progressed = true;
            }
            if (jq < nt && ready(full_bar(jq % kPtRing), static_cast<uint32_t>((jq / kPtRing) & 1)) &&
                (jq < 2 || ready(sfree_bar(jq & 1), static_cast<uint32_t>(((jq - 2) >> 1) & 1)))) {
                if (jq > 0 && (jq % (32 / BPS)) == 0) {
                    ecur = enext;
                    enext = load_entry((jq / (32 / BPS) + 1) * 32 + lane);
                }
                const uint32_t st = sbase + (jq % kPtRing) * C::STAGE;
                // value rows of keys past the row's end or in a block whose entry is bad: zero
                const int key0 = jq * kPtKeys;
                const int blk = jq * BPS + (lane & (BPS - 1));
                const int32_t e = __shfl_sync(kFull, ecur, (jq % (32 / BPS)) * BPS + (lane & (BPS - 1)));
                const bool bv = blk < nblk && e >= 0 && static_cast<int64_t>(e) < p.N;
                const uint32_t vmask = __ballot_sync(kFull, bv) & ((1u << BPS) - 1u);
                if (key0 + kPtKeys > total || vmask != (1u << BPS) - 1u) {
                    for (int i = lane; i < kPtKeys * 8 * C::BANDS; i += 32) {
                        const int row = i / (8 * C::BANDS), c = i % (8 * C::BANDS);
                        if (key0 + row >= total || !(vmask >> (row >> 4) & 1u))
                            sts128_zero(st + (C::BANDS + (c >> 3)) * C::KBAND + sw128(row, c & 7));
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                tc_fence_after();
                {
                    const uint64_t b0 = tc_smem_desc(st, 16, 1024, kSwizzle128B);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk)   // 16 channels (32 bytes) per MMA, 4 per 128-byte band
                        tc_mma_f16_warp(tmem + (jq & 1) * kPtKeys,
                                        tc_desc_advance(desc_q, (kk >> 2) * C::QBAND + (kk & 3) * 32),
                                        tc_desc_advance(b0, (kk >> 2) * C::KBAND + (kk & 3) * 32), idesc_qk,
                                        kk > 0 ? 1u : 0u);
                    tc_commit_warp(sfull_bar(jq & 1));
                }
                __syncwarp();
                ++jq;
                progressed = true;
            }
            if (progressed) {
                idle = 0;
                idle_since = 0;
            } else if ((++idle & 63u) == 0u) {   // bounded: 2 s without progress is an expired wait
                const uint64_t now = globaltimer_ns();
                if (idle_since == 0) idle_since = now;
                else if (now - idle_since > 2000000000ull) {
                    timed_out = true;
                    break;
                }
            }
        }
    } else if (warp < 4) {
        // ------------------------------------------------------------ softmax: thread = query row
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const int pos = pos0 + tid / g;
        const int vis = min(q_start + pos + 1, total);   // keys this row may read (rows past the chunk: all)
        float m = -INFINITY, l = 0.f;
        int j = 0;
        for (; j < nt; ++j) {
            const int sb = j & 1;
            const bool ok1 = mbar_wait_bounded(sfull_bar(sb), static_cast<uint32_t>((j >> 1) & 1));
            tc_fence_after();
            uint32_t r0[32], r1[32];
            tmem_ld32(tmem + sb * kPtKeys + lane_off, r0);
            tmem_ld32(tmem + sb * kPtKeys + 32 + lane_off, r1);
            tmem_ld_wait(r0);
            tmem_ld_wait(r1);
            tc_fence_before();
            mbar_arrive(sfree_bar(sb));

            // keys past the row's visible end (the causal diagonal, or the row's end) count
            // nothing; stages wholly visible to the row skip the masking
            const int nvis = vis - j * kPtKeys;
            float sv[64];
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                sv[c] = __uint_as_float(r0[c]);
                sv[32 + c] = __uint_as_float(r1[c]);
            }
            if (nvis < kPtKeys) {
#pragma unroll
                for (int c = 0; c < 64; ++c) sv[c] = c < nvis ? sv[c] : -INFINITY;
            }
            float b0 = sv[0], b1 = sv[1], b2 = sv[2], b3 = sv[3];   // four chains of 3-input maxima
#pragma unroll
            for (int c = 4; c < 60; c += 8) {
                b0 = max3f(b0, sv[c], sv[c + 1]);
                b1 = max3f(b1, sv[c + 2], sv[c + 3]);
                b2 = max3f(b2, sv[c + 4], sv[c + 5]);
                b3 = max3f(b3, sv[c + 6], sv[c + 7]);
            }
            b0 = max3f(b0, sv[60], sv[61]);
            b1 = max3f(b1, sv[62], sv[63]);
            float bm = max3f(b0, b1, fmaxf(b2, b3));
            bm *= p.scale_log2;                           // scale > 0: the max of the scaled scores
            const bool move = bm > m + kRescaleSlack;   // the first visible key always moves a -inf maximum
            float alpha = 1.f;
            if (move) {
                alpha = fast_exp2(m - bm);              // 0 while nothing was visible
                m = bm;
                l *= alpha;
            }
            // the warp rescales its O rows together, once the value MMA of stage j - 1 is in O
            const bool rescale = j > 0 && __any_sync(kFull, move && alpha != 1.f);
            const bool ok3 = !rescale || mbar_wait_bounded(pvdone_bar((j - 1) & 1), static_cast<uint32_t>(((j - 1) >> 1) & 1));
            if (rescale && ok3) {
                tc_fence_after();
#pragma unroll
                for (int part = 0; part < D / 32; ++part) {
                    uint32_t o[32];
                    tmem_ld32(tm_o + part * 32 + lane_off, o);
                    tmem_ld_wait(o);
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                    tmem_st32(tm_o + part * 32 + lane_off, o);
                }
                tmem_st_wait();
            }
            // weights 2^(scale s - m): m is finite from the first stage on (key 0 is visible to
            // every row), and a masked score (-inf) weighs 0
            const float neg_m = -m;
            uint32_t pk[32];
            float ls[4] = {0.f, 0.f, 0.f, 0.f};   // four partial sums: short dependency chains
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
                const float p0 = fast_exp2(fmaf(sv[c], p.scale_log2, neg_m));
                const float p1 = fast_exp2(fmaf(sv[c + 1], p.scale_log2, neg_m));
                ls[(c / 2) & 3] += p0 + p1;
                pk[c / 2] = pack_bf16(p0, p1);
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            // the value MMA of stage j - 2 has read this stage's weight buffer (waited for only
            // now, behind the exponentials)
            const bool ok2 = j < 2 || mbar_wait_bounded(pvdone_bar(j & 1), static_cast<uint32_t>(((j - 2) >> 1) & 1));
            if (!softmax_all(ok1 && ok2 && ok3)) {   // one CTA-wide vote per stage: a wait expired anywhere
                timed_out = true;
                break;
            }
#pragma unroll
            for (int c = 0; c < 8; ++c)
                sts128(sbase + C::P + (j & 1) * (128 * 128) + sw128(tid, c),
                       make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(pfull_bar(j & 1));
        }

        bool ok = !timed_out &&
                  mbar_wait_bounded(pvdone_bar((nt - 1) & 1), static_cast<uint32_t>(((nt - 1) >> 1) & 1));
        ok = softmax_all(ok);
        if (!ok) {
            timed_out = true;
        } else {
            tc_fence_after();
            const bool real = pos < n_q;
            const size_t orow = (static_cast<size_t>(pos) * p.H_Q + h * g + tid % g);
            const float inv = 1.f / l;
#pragma unroll
            for (int part = 0; part < D / 32; ++part) {
                uint32_t o[32];
                tmem_ld32(tm_o + part * 32 + lane_off, o);
                tmem_ld_wait(o);
                if (real) {
                    float4 *dst = reinterpret_cast<float4 *>(p.out + orow * D + part * 32);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        dst[c] = make_float4(__uint_as_float(o[4 * c]) * inv, __uint_as_float(o[4 * c + 1]) * inv,
                                             __uint_as_float(o[4 * c + 2]) * inv, __uint_as_float(o[4 * c + 3]) * inv);
                }
            }
            if (real && p.lse) p.lse[orow] = (m + log2f(l)) * kLn2;
        }
    }
    if (timed_out && lane == 0) atomicOr(p.err, KVC_EBIT_TIMEOUT);

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, C::COLS);
    }
}

// grid (1, KV head, tile of 128 / g positions), 224 threads.  Launched as a
// programmatic dependent in the mixed step: it reads only the chunk's row,
// which the step before it does not write, so it never waits on that step.
template <int D>
__global__ void __launch_bounds__(kPtThreads, 1) prefill_tc_kernel(const __grid_constant__ CUtensorMap tmap16,
                                                                    const DecodeParams p)
{
    prefill_tc_cta<D>(tmap16, p, blockIdx.z, blockIdx.y);
}

// The tensor-memory prefill kernel for a pool (fn = nullptr: d_h 64 / 128 bf16 pools only).
DecodeKernel select_prefill_tc(int D, int dtype);

}  // namespace kvc
