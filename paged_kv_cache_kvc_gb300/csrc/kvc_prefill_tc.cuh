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
// heads.
//
// The CTA's keys (64 per stage) are split into two streams, stream 0 the first
// half of its stages and stream 1 the rest, each with its own staging ring,
// score, weight and output accumulators in TMEM and softmax warps; the epilogue merges
// the two partial softmaxes of every row (the log-sum-exp merge of split
// attention).  One stream's chain of score MMA -> softmax -> value MMA leaves
// the tensor cores and the single MMA-issuing thread idle most of the time;
// two independent chains fill each other's gaps.  384 threads:
//   warps 8, 9    TMA producers of stream 0 and 1: per stage the key rows and
//                 value rows of its 4 blocks, one 16-row box per block, 128-byte
//                 band and keys / values (128-byte swizzle), a ring of 3 stages.
//   warps 10, 11  MMA issuers of stream 0 and 1 (one elected lane each; the
//                 issue of an MMA holds its thread while the pipe takes it, so
//                 one thread per stream), per stage:
//                   S[128 x 64]  = Q[128 x D] . K^T        (K-major A and B)
//                   O[128 x D]  += P[128 x 64] . V[64 x D]  (A from TMEM, MN-major B)
//                 S double-buffered per stream in TMEM; the softmax writes P as
//                 bf16 pairs over the first 32 columns of its own S buffer, so
//                 the buffer is reused by the score MMA two stages later only
//                 after the value MMA has read P.
//   warps 0..3    softmax of stream 0, warps 4..7 of stream 1; thread = query
//                 row (TMEM lane): the causal mask (key < q_start + position +
//                 1), the row's running maximum as a reference that moves only
//                 when a score exceeds it by more than 8 (log2 units), then the
//                 row's O and sum are rescaled (the warp together, after the
//                 stream's previous value MMA has landed); P row as bf16 into
//                 TMEM.
// Value rows of keys past the row's end or of blocks not loaded are zeroed
// before the value MMA (a zero weight times NaN is NaN).  The epilogue merges
// the streams with weights 2^(m_s - max m) and divides by the merged sum.
#pragma once
#include "kvc_decode_tc.cuh"

namespace kvc {

constexpr int kPtKeys = 64;                     // keys per stage
constexpr int kPtRing = 3;                      // stages in flight per stream
constexpr int kPtThreads = 384;

template <int D>
struct PrefillTcCfg {
    static constexpr int BANDS = D / 64;                      // 128-byte column bands of a bf16 row
    static constexpr int KBAND = kPtKeys * 128;               // one band of the stage's 64 key rows
    static constexpr int STAGE = 2 * BANDS * KBAND;           // keys, then values
    static constexpr int QBAND = 128 * 128;                   // one band of the 128 query rows
    static constexpr int Q = 0;
    static constexpr int RING = Q + BANDS * QBAND;            // [stream][slot] stages
    static constexpr int BARS = RING + 2 * kPtRing * STAGE;
    // per stream: full[R], kvfree[R], s_full[2], p_full[2], pv_done[2]
    static constexpr int BARS_PER_STREAM = 2 * kPtRing + 6;
    static constexpr int VMASK = BARS + 2 * BARS_PER_STREAM * 8;   // [stream][slot] loaded-block masks
    static constexpr int ABORT = VMASK + 2 * kPtRing * 4;          // set when a wait expires anywhere
    static constexpr int XCH = ABORT + 8;                          // stream 1's (m, l) per row for the merge
    static constexpr int SLOT = XCH + 128 * 8;
    static constexpr int SMEM = 1024 + SLOT + 16;
    static constexpr uint32_t COLS = 512;   // stream s: S/P[0] s*256 + 0..63, S/P[1] + 64..127, O from s*256 + 128
};

// A vote of the 128 threads of one softmax group (named barrier `id`).
__device__ __forceinline__ bool group_all(bool v, uint32_t id)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, 128, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"(v ? 1u : 0u), "r"(id)
                 : "memory");
    return r != 0;
}

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
    // stream 0: stages [0, split), stream 1: [split, nt) (empty when nt == 1)
    const int split = (nt + 1) / 2;
    auto s_begin = [&](int s) { return s == 0 ? 0 : split; };
    auto s_count = [&](int s) { return s == 0 ? split : nt - split; };

    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + C::BARS;
    auto sbar = [&](int s, int i) { return bars + 8u * (s * C::BARS_PER_STREAM + i); };
    auto full_bar = [&](int s, int r) { return sbar(s, r); };
    auto kvfree_bar = [&](int s, int r) { return sbar(s, kPtRing + r); };
    auto sfull_bar = [&](int s, int b) { return sbar(s, 2 * kPtRing + b); };
    auto pfull_bar = [&](int s, int b) { return sbar(s, 2 * kPtRing + 2 + b); };
    auto pvdone_bar = [&](int s, int b) { return sbar(s, 2 * kPtRing + 4 + b); };
    auto stage_addr = [&](int s, int r) { return sbase + C::RING + (s * kPtRing + r) * C::STAGE; };
    volatile uint32_t *vmask_sh = reinterpret_cast<volatile uint32_t *>(smem + C::VMASK);
    volatile uint32_t *abort_sh = reinterpret_cast<volatile uint32_t *>(smem + C::ABORT);
    float2 *xch = reinterpret_cast<float2 *>(smem + C::XCH);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::SLOT);

    if (tid == 0) {
        for (int s = 0; s < 2; ++s) {
            for (int r = 0; r < kPtRing; ++r) {
                mbar_init(full_bar(s, r), 1);
                mbar_init(kvfree_bar(s, r), 1);
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(sfull_bar(s, b), 1);
                mbar_init(pfull_bar(s, b), 128);
                mbar_init(pvdone_bar(s, b), 1);
            }
        }
        fence_barrier_init();
        prefetch_tensormap(&tmap16);
        *abort_sh = 0u;
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), C::COLS);
        tmem_relinquish();
    }
    // the query rows (zero past the chunk), the K-major A operand of the score MMA: row r is
    // position pos0 + r / g, head h g + r mod g; consecutive threads take consecutive 16-byte
    // chunks of a row, so a warp reads whole rows (g rows of a position are contiguous)
#pragma unroll 2
    for (int x = tid; x < 128 * (D / 8); x += kPtThreads) {
        const int r = x / (D / 8), c = x % (D / 8), pos = pos0 + r / g;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (pos < n_q)
            v = *reinterpret_cast<const uint4 *>(p.q + (static_cast<size_t>(pos) * p.H_Q + h * g + r % g) * D + c * 8);
        sts128(sbase + C::Q + (c >> 3) * C::QBAND + sw128(r, c & 7), v);
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    constexpr int BPS = kPtKeys / kBS;                // blocks per stage
    constexpr int SPW = 32 / BPS;                     // stages per 32-entry table window
    auto load_entry = [&](int blk) -> int32_t { return blk < nblk ? __ldg(p.bt + blk) : -1; };

    bool timed_out = false;
    if (warp == 8 || warp == 9) {
        // ------------------------------------------------------------ TMA producer of stream s
        const int s = warp - 8, b = s_begin(s), n = s_count(s);
        // lane l holds entry 32 w + l of table window w (the stages of window w: SPW w .. SPW w + SPW - 1)
        int w = b / SPW;
        int32_t ecur = load_entry(32 * w + lane), enext = load_entry(32 * (w + 1) + lane);
        const int nload = p.stall_loads ? 0 : n;   // the test hook withholds every load
        int i = 0;
        for (; i < nload; ++i) {
            const int j = b + i, r = i % kPtRing;
            if (j / SPW != w) {
                ++w;
                ecur = enext;
                enext = load_entry(32 * (w + 1) + lane);
            }
            if (i >= kPtRing) {
                const bool ok = mbar_wait_bounded(kvfree_bar(s, r), static_cast<uint32_t>(((i / kPtRing) - 1) & 1));
                if (!__all_sync(kFull, ok)) {
                    if (lane == 0) *abort_sh = 1u;
                    timed_out = true;
                    break;
                }
            }
            const int blk = j * BPS + lane;
            const int32_t e = __shfl_sync(kFull, ecur, (j % SPW) * BPS + (lane & (BPS - 1)));
            const bool v = lane < BPS && blk < nblk && e >= 0 && static_cast<int64_t>(e) < p.N;
            if (lane < BPS && blk < nblk && !v) atomicOr(p.err, KVC_EBIT_BAD_BLOCK);
            const uint32_t mask = __ballot_sync(kFull, v) & ((1u << BPS) - 1u);
            if (lane == 0) {
                vmask_sh[s * kPtRing + r] = mask;   // published by the arrive below
                if (mask == 0u) mbar_arrive(full_bar(s, r));
                else
                    mbar_arrive_expect_tx(full_bar(s, r),
                                          static_cast<uint32_t>(__popc(mask)) * 2u * C::BANDS * (kBS * 128u));
            }
            __syncwarp();
            // one box per lane, all in one instruction: lane = (band, keys / values, block);
            // every lane already holds the entry of block lane mod BPS
            const int bl = lane % BPS, kvp = (lane / BPS) & 1, band = lane / (2 * BPS);
            if (lane < 2 * BPS * C::BANDS && ((mask >> bl) & 1u)) {
                const int32_t y = static_cast<int32_t>(((row_layer + e) * p.H_KV + h) * (2 * kBS)) + kvp * kBS;
                tma_load_2d(stage_addr(s, r) + (kvp * C::BANDS + band) * C::KBAND + bl * (kBS * 128), &tmap16,
                            full_bar(s, r), band * 64, y);
            }
        }
        // before the CTA exits: the copies of the last slots have landed and their releases
        // are in (immediate unless a wait expired)
        if (lane == 0)
            for (int ii = max(0, i - kPtRing); ii < i; ++ii) {
                (void)mbar_wait_bounded(full_bar(s, ii % kPtRing), static_cast<uint32_t>((ii / kPtRing) & 1),
                                        100000000ull);
                (void)mbar_wait_bounded(kvfree_bar(s, ii % kPtRing), static_cast<uint32_t>((ii / kPtRing) & 1),
                                        100000000ull);
            }
        __syncwarp();
    } else if (warp == 10 || warp == 11) {
        // ------------------------------------------------------------ MMA issuer of stream warp - 10
        constexpr uint32_t idesc_qk = tc_idesc_f16(128, kPtKeys, true, false, false);
        constexpr uint32_t idesc_pv = tc_idesc_f16(128, D, true, false, true);
        // Issues whichever MMA of its stream is ready: the value MMA of a stage
        // once its weights are in TMEM (it releases the stage), the score MMA of a stage once
        // its keys have landed and the value MMA two stages back has read the weights in its
        // score buffer.  Barriers are tested without blocking, lane 0 testing for the warp.
        auto ready = [&](uint32_t bar, uint32_t parity) {
            const uint32_t r = lane == 0 ? (mbar_test_wait(bar, parity) ? 1u : 0u) : 0u;
            return __shfl_sync(kFull, r, 0) != 0u;
        };
        const uint64_t desc_q = tc_smem_desc(sbase + C::Q, 16, 1024, kSwizzle128B);
        const int s = warp - 10, n = s_count(s);
        const uint32_t tm_s = tmem + s * 256;
        int jq = 0, jp = 0;
        uint64_t idle_since = 0;
        uint32_t idle = 0;
        while (jp < n) {
            bool progressed = false;
            if (jp < jq && ready(pfull_bar(s, jp & 1), static_cast<uint32_t>((jp >> 1) & 1))) {
                const int i = jp;
                tc_fence_after();
                const uint64_t b0 = tc_smem_desc(stage_addr(s, i % kPtRing) + C::BANDS * C::KBAND, C::KBAND, 1024,
                                                 kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < kPtKeys / 16; ++kk)   // 16 keys: 8 TMEM columns of P, 2048 bytes of V rows
                    tc_mma_f16_tmem_a_warp(tm_s + 128, tm_s + (i & 1) * kPtKeys + kk * 8,
                                           tc_desc_advance(b0, kk * 2048), idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
                tc_commit_warp(kvfree_bar(s, i % kPtRing));
                tc_commit_warp(pvdone_bar(s, i & 1));
                __syncwarp();
                ++jp;
                progressed = true;
            }
            if (jq < n && ready(full_bar(s, jq % kPtRing), static_cast<uint32_t>((jq / kPtRing) & 1)) &&
                (jq < 2 ||
                 (jq - 2 < jp &&
                  ready(pvdone_bar(s, jq & 1), static_cast<uint32_t>(((jq - 2) >> 1) & 1))))) {
                const int i = jq, j = s_begin(s) + i, key0 = j * kPtKeys;
                const uint32_t st = stage_addr(s, i % kPtRing);
                // value rows of keys past the row's end or of blocks not loaded: zero
                const uint32_t vmask = vmask_sh[s * kPtRing + i % kPtRing];
                if (key0 + kPtKeys > total || vmask != (1u << BPS) - 1u) {
                    for (int x = lane; x < kPtKeys * 8 * C::BANDS; x += 32) {
                        const int row = x / (8 * C::BANDS), c = x % (8 * C::BANDS);
                        if (key0 + row >= total || !(vmask >> (row >> 4) & 1u))
                            sts128_zero(st + (C::BANDS + (c >> 3)) * C::KBAND + sw128(row, c & 7));
                    }
                    fence_proxy_async_smem();
                }
                __syncwarp();
                tc_fence_after();
                const uint64_t b0 = tc_smem_desc(st, 16, 1024, kSwizzle128B);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk)   // 16 channels (32 bytes) per MMA, 4 per 128-byte band
                    tc_mma_f16_warp(tm_s + (i & 1) * kPtKeys,
                                    tc_desc_advance(desc_q, (kk >> 2) * C::QBAND + (kk & 3) * 32),
                                    tc_desc_advance(b0, (kk >> 2) * C::KBAND + (kk & 3) * 32), idesc_qk,
                                    kk > 0 ? 1u : 0u);
                tc_commit_warp(sfull_bar(s, i & 1));
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
                if (__any_sync(kFull, *abort_sh != 0u) || now - idle_since > 2000000000ull) {
                    if (lane == 0) *abort_sh = 1u;
                    timed_out = true;
                    break;
                }
            }
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------ softmax of stream s: thread = query row
        const int s = warp >> 2, row = tid & 127, b = s_begin(s), n = s_count(s);
        const uint32_t vote_id = 1u + static_cast<uint32_t>(s);
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tm_s = tmem + s * 256, tm_o = tm_s + 128;
        const int pos = pos0 + row / g;
        const int vis = min(q_start + pos + 1, total);   // keys this row may read (rows past the chunk: all)
        float m = -INFINITY, l = 0.f;
        int i = 0;
        for (; i < n; ++i) {
            const int j = b + i, sb = i & 1;
            if (__any_sync(kFull, *abort_sh != 0u)) {   // a wait expired elsewhere in the CTA
                timed_out = true;
                break;
            }
            const bool ok1 = mbar_wait_bounded(sfull_bar(s, sb), static_cast<uint32_t>((i >> 1) & 1));
            tc_fence_after();
            uint32_t r0[32], r1[32];
            tmem_ld32(tm_s + sb * kPtKeys + lane_off, r0);
            tmem_ld32(tm_s + sb * kPtKeys + 32 + lane_off, r1);
            tmem_ld_wait(r0);
            tmem_ld_wait(r1);

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
            bm *= p.scale_log2;                         // scale > 0: the max of the scaled scores
            const bool move = bm > m + kRescaleSlack;   // -inf (nothing visible yet) never moves
            float alpha = 1.f;
            if (move) {
                alpha = fast_exp2(m - bm);              // 0 while nothing was visible
                m = bm;
                l *= alpha;
            }
            // the warp rescales its O rows together, once the stream's previous value MMA is in O
            const bool rescale = i > 0 && __any_sync(kFull, move && alpha != 1.f);
            const bool ok3 = !rescale || mbar_wait_bounded(pvdone_bar(s, (i - 1) & 1),
                                                           static_cast<uint32_t>(((i - 1) >> 1) & 1));
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
            // weights 2^(scale s - m); a masked score (-inf) weighs 0, and so does every key
            // while none has been visible to the row (m = -inf: stream 1 can start past the
            // causal end of a row at the tile's start)
            const float neg_m = m == -INFINITY ? 0.f : -m;
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
            // a wait expired: the warp leaves the loop together and tells the others, which leave
            // theirs at their next stage (their waits are bounded); the group's vote below
            // gathers the warps again
            if (!__all_sync(kFull, ok1 && ok3)) {
                if (lane == 0) *abort_sh = 1u;
                timed_out = true;
                break;
            }
            // P row over the first 32 columns of this stage's score buffer (its scores are in
            // registers): the A operand of the value MMA
            tmem_st32(tm_s + sb * kPtKeys + lane_off, pk);
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(pfull_bar(s, sb));
        }

        bool ok = !timed_out && (n == 0 || mbar_wait_bounded(pvdone_bar(s, (n - 1) & 1),
                                                             static_cast<uint32_t>(((n - 1) >> 1) & 1)));
        ok = group_all(ok, vote_id);
        if (!ok) timed_out = true;
        if (s == 1) {
            // stream 1 hands its (m, l) to stream 0's thread of the same row; l < 0 marks an
            // expired wait (its O must not be read)
            xch[row] = make_float2(m, ok ? l : -1.f);
            asm volatile("bar.arrive 3, 256;" ::: "memory");
        } else {
            asm volatile("bar.sync 3, 256;" ::: "memory");
            const float2 o1 = xch[row];
            const bool use1 = s_count(1) > 0 && o1.x != -INFINITY;   // stream 1 saw keys of this row
            const int n1 = s_count(1);   // stream 1's last value MMA, observed here too before its O is read
            const bool ok1 = n1 == 0 || o1.y < 0.f ||
                             mbar_wait_bounded(pvdone_bar(1, (n1 - 1) & 1),
                                               static_cast<uint32_t>(((n1 - 1) >> 1) & 1));
            if (ok && ok1 && o1.y >= 0.f) {
                tc_fence_after();
                const float M = use1 ? fmaxf(m, o1.x) : m;   // m is finite: key 0 is visible to every row
                const float w0 = fast_exp2(m - M), w1 = use1 ? fast_exp2(o1.x - M) : 0.f;
                const float L = w0 * l + w1 * o1.y;
                const bool real = pos < n_q;
                const size_t orow = (static_cast<size_t>(pos) * p.H_Q + h * g + row % g);
                const float a0 = w0 / L, a1 = w1 / L;
#pragma unroll
                for (int part = 0; part < D / 32; ++part) {
                    uint32_t o[32], u[32];
                    tmem_ld32(tm_o + part * 32 + lane_off, o);
                    tmem_ld_wait(o);
                    if (s_count(1) > 0) {   // uniform: stream 1's O exists (finite: zero weights x finite rows)
                        tmem_ld32(tmem + 256 + 128 + part * 32 + lane_off, u);
                        tmem_ld_wait(u);
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c) u[c] = 0u;
                    }
                    if (real) {
                        float4 *dst = reinterpret_cast<float4 *>(p.out + orow * D + part * 32);
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            float4 v;
                            v.x = fmaf(__uint_as_float(o[4 * c]), a0, __uint_as_float(u[4 * c]) * a1);
                            v.y = fmaf(__uint_as_float(o[4 * c + 1]), a0, __uint_as_float(u[4 * c + 1]) * a1);
                            v.z = fmaf(__uint_as_float(o[4 * c + 2]), a0, __uint_as_float(u[4 * c + 2]) * a1);
                            v.w = fmaf(__uint_as_float(o[4 * c + 3]), a0, __uint_as_float(u[4 * c + 3]) * a1);
                            dst[c] = v;
                        }
                    }
                }
                if (real && p.lse) p.lse[orow] = (M + log2f(L)) * kLn2;
            } else {
                timed_out = true;
            }
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

// grid (1, KV head, tile of 128 / g positions), 384 threads.  Launched as a
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
