// Paged decode attention for 32-head groups (MQA) on e4m3 pools, on the
// fifth-generation tensor cores: the same computation as the split kernel's
// e4m3 path ("KV cache: Generation state, latency, and allocation" 21.1 and
// 21.5; the FP8 KV-cache page: a per-channel scale per (layer, KV head)), laid
// out as the bf16 tensor-memory kernel (thread = token softmax, scores and
// outputs in TMEM).
//
// The tensor cores take no e4m3 operand against bf16 queries, so the codes are
// staged by TMA and widened to f16 (exact: every e4m3 value is an f16 value).
// The key scale s_K is folded into the queries (q_c s_K,c, rounded to f16) and
// the value scale s_V into the output (o_c s_V,c), as in the split kernel.  The
// widening runs on the ALU pipe of every SM sub-partition, each stage is
// double-buffered so that the value MMA of one tile overlaps the softmax of the
// next, and each role has warps of its own (a single warp per sub-partition
// runs a latency-bound chain).  384 threads, three warpgroups; the softmax
// warpgroup takes 240 registers a thread, the other two 128 (setmaxnreg; 63 488
// of the 64 512 allocated at launch):
//   warps 0..3  softmax, thread t = token t of the tile.
//   warp 4      TMA producer: a tile's 8 blocks, each one 32-row box of codes
//               (keys in rows 0..15, values 16..31, 128-byte swizzle), a ring of
//               3 tiles of codes (96 KB in flight per SM).
//   warp 5      MMA issuer: S^T[128 tok x 32] = K . Q^T with K from tensor memory,
//               O^T[128 ch x 64] += V^T . P^T (high and low f16 parts of each
//               weight).
//   warps 6, 7  value converters: 64 positions each into one of two f16 value
//               tiles in shared memory (the layout the MMA descriptor names), rows
//               that must not count written as zeros, the step's own value row
//               quantised, written to the pool and used.
//   warps 8..11 key wideners, thread t = token 32 (warp - 8) + t: its key row into
//               tensor memory (the A operand of the score MMA: lane t, f16 pairs in
//               64 columns, two buffers); the warp that holds the step's own
//               position quantises its key row (fused append), writes it to the
//               pool and uses it.
#pragma once
#include "kvc_decode_tc.cuh"

namespace kvc {

constexpr int kT8Threads = 384;
constexpr int kT8Ring = 3;                                // tiles of codes in flight
constexpr int kT8CodeSlot = kTcBlocks * 2 * kBS * 128;    // 8 blocks x 32 rows x 128 B = 32 KiB
constexpr int kT8VF = kT8Ring * kT8CodeSlot;              // 2 f16 value tiles: 2 bands x 128 rows x 128 B each
constexpr int kT8Q = kT8VF + 2 * kTcSlot;                 // Q (f16, s_K folded): 2 bands x 32 rows x 128 B
constexpr int kT8P = kT8Q + 2 * 32 * 128;                 // 2 x P^T: 128 token rows x 64 f16
constexpr int kT8Bars = kT8P + 2 * kTcTok * 128;
// barriers: code_full[R], code_free[R], kf_full[2], s_full[2], s_free[2], pv_ready[2], pv_done[2], q_ready
constexpr int kT8NumBars = 2 * kT8Ring + 11;
constexpr int kT8Vmask = kT8Bars + ((kT8NumBars * 8 + 15) & ~15);   // [R] loaded-block masks
constexpr int kT8Red = kT8Vmask + 16;                               // float [4][32], msh, ash, lsh
constexpr int kT8TmemSlot = kT8Red + (4 * 32 + 3 * 32) * 4;
constexpr int kT8Smem = 1024 + kT8TmemSlot + 16;
// TMEM: S[0] 0..31, S[1] 32..63, O^T 64..127 (high part, then low part), K[0] 128..191, K[1] 192..255
constexpr uint32_t kT8Cols = 256;

// Register shares of a warpgroup (all its threads execute these): the softmax warpgroup takes
// 240 a thread, the two others give theirs down to 128.  Launch: 384 threads x 168 = 64 512.
__device__ __forceinline__ void regs_up_240() { asm volatile("setmaxnreg.inc.sync.aligned.u32 240;" ::: "memory"); }
__device__ __forceinline__ void regs_down_128() { asm volatile("setmaxnreg.dec.sync.aligned.u32 128;" ::: "memory"); }

// 16 e4m3 codes (one 16-byte chunk) to 16 f16 values: 8 words, word i = channels 2 i (low half), 2 i + 1
__device__ __forceinline__ void e4m3x16_to_f16(const uint4 &w, uint32_t *o)
{
    e4m3x4_to_f16x2x2(w.x, o[0], o[1]);
    e4m3x4_to_f16x2x2(w.y, o[2], o[3]);
    e4m3x4_to_f16x2x2(w.z, o[4], o[5]);
    e4m3x4_to_f16x2x2(w.w, o[6], o[7]);
}

// Four channels of the step's own row (bf16, 8 bytes at src), quantised with their scales
// (round to nearest e4m3, saturating), as in the split kernel's fused append.
__device__ __forceinline__ uint32_t quantize4_e4m3(const uint16_t *src, const float *sc)
{
    const uint2 x = *reinterpret_cast<const uint2 *>(src);
    const float f[4] = {bf16_lo(x.x), bf16_hi(x.x), bf16_lo(x.y), bf16_hi(x.y)};
    uint32_t q = 0u;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        q |= static_cast<uint32_t>(__nv_cvt_float_to_fp8(__fdiv_rn(f[i], __ldg(sc + i)), __NV_SATFINITE, __NV_E4M3))
             << (8 * i);
    return q;
}

// One split of unit (b, h), G = 32 query heads, e4m3 pool, d_h 128.
template <int G>
__device__ __forceinline__ void decode_tc8_cta(const CUtensorMap &tmap, const DecodeParams &p, const int split,
                                               const int h, const int b)
{
    static_assert(G == 32, "the TMEM score buffers and the head reductions are laid out for 32 heads");
    constexpr int D = 128;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hq0 = h * p.g;

    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + kT8Bars;
    auto code_full = [&](int s) { return bars + 8u * s; };
    auto code_free = [&](int s) { return bars + 8u * (kT8Ring + s); };
    auto kf_full = [&](int kb) { return bars + 8u * (2 * kT8Ring + kb); };
    auto sfull_bar = [&](int sb) { return bars + 8u * (2 * kT8Ring + 2 + sb); };
    auto sfree_bar = [&](int sb) { return bars + 8u * (2 * kT8Ring + 4 + sb); };
    auto pvready_bar = [&](int pb) { return bars + 8u * (2 * kT8Ring + 6 + pb); };
    auto pvdone_bar = [&](int pb) { return bars + 8u * (2 * kT8Ring + 8 + pb); };
    const uint32_t qready_bar = bars + 8u * (2 * kT8Ring + 10);
    volatile uint32_t *vmask_sh = reinterpret_cast<volatile uint32_t *>(smem + kT8Vmask);
    float *red = reinterpret_cast<float *>(smem + kT8Red);   // [4][32]
    float *msh = red + 128, *ash = msh + 32, *lsh = ash + 32;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kT8TmemSlot);

    // ---- set-up, before any global memory access
    if (tid == 0) {
        for (int s = 0; s < kT8Ring; ++s) {
            mbar_init(code_full(s), 1);
            mbar_init(code_free(s), 6);   // the 4 key wideners and the 2 value converters
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(kf_full(i), 128);
            mbar_init(sfull_bar(i), 1);
            mbar_init(sfree_bar(i), 128);
            mbar_init(pvready_bar(i), 128 + 2);   // the weights (128 threads) and the values (2 warps)
            mbar_init(pvdone_bar(i), 1);
        }
        mbar_init(qready_bar, 128);
        fence_barrier_init();
        prefetch_tensormap(&tmap);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kT8Cols);
        tmem_relinquish();
    }
    if (tid < 32) msh[tid] = -INFINITY;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // launched as a programmatic dependent: the set-up above overlaps the kernel before it
    grid_dependency_wait();

    int len = seq_len(p, b);
    if (len < 0 || static_cast<int64_t>(len) > static_cast<int64_t>(p.max_blocks) * kBS) {
        if (split == 0 && tid == 0) atomicOr(p.err, KVC_EBIT_RANGE);
        len = 0;
    }
    const int nblk = (len + kBS - 1) / kBS;
    if (nblk == 0 && split == 0) {   // empty sequence: zero output, lse = -inf
        for (int i = tid; i < G * D; i += kT8Threads) p.out[(static_cast<size_t>(b) * p.H_Q + hq0) * D + i] = 0.f;
        if (p.lse && tid < G) p.lse[static_cast<size_t>(b) * p.H_Q + hq0 + tid] = -INFINITY;
    }
    // split: blocks blk0 .. blk_end - 1, walked as 128-token tiles from blk0 (the last one may be partial;
    // blocks past blk_end belong to the next split and count here as unstaged)
    const int blk0 = split * p.chunk;
    if (blk0 < nblk) {   // uniform over the CTA: this split holds blocks
        const int blk_end = min(nblk, blk0 + p.chunk);
        const int nt = (blk_end - blk0 + kTcBlocks - 1) / kTcBlocks;
        const int ns = (nblk + p.chunk - 1) / p.chunk;
        const int32_t *bt_row = p.bt + static_cast<int64_t>(b) * p.bt_stride;
        const int64_t row_layer = static_cast<int64_t>(p.layer) * p.N;
        const float *s_k = p.s_k + static_cast<size_t>(h) * D, *s_v = p.s_v + static_cast<size_t>(h) * D;

        if (tid < 128) {   // q rows times s_K, as f16 (K-major B operand of the score MMA)
            for (int i = tid; i < G * 16; i += 128) {   // row hh, 8-channel chunk c of 16
                const int hh = i >> 4, c = i & 15;
                const uint4 v = *reinterpret_cast<const uint4 *>(p.q + (static_cast<size_t>(b) * p.H_Q + hq0 + hh) * D +
                                                                 c * 8);
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                uint32_t o[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    o[k] = pack_f16(bf16_lo(w[k]) * __ldg(s_k + c * 8 + 2 * k),
                                    bf16_hi(w[k]) * __ldg(s_k + c * 8 + 2 * k + 1));
                sts128(sbase + kT8Q + (c >> 3) * (32 * 128) + sw128(hh, c & 7), make_uint4(o[0], o[1], o[2], o[3]));
            }
            fence_proxy_async_smem();
            mbar_arrive(qready_bar);
        }
        const uint32_t tm_o = tmem + 64, tm_k = tmem + 128;

        bool timed_out = false;
        const int bbase = blk0;
        auto load_entry = [&](int rel) -> int32_t { return bbase + rel < blk_end ? __ldg(bt_row + bbase + rel) : -1; };
        // the step's own position (fused append); it lies in this split if it is in one of its tiles
        const int app = p.k_new ? len - 1 : -1;
        const int32_t app_phys = app >= 0 ? __ldg(bt_row + app / kBS) : -1;   // valid where its block is loaded

        // the register shares are set at the top of each warpgroup's branch, so that the code of the branch
        // is compiled against its own share
        if (warp >= 4 && warp < 8) {
            regs_down_128();
            if (warp == 4) {
                // ------------------------------------------------------------ TMA producer (codes)
                int32_t ecur = load_entry(lane), enext = load_entry(32 + lane);
                const int nload = p.stall_loads ? 0 : nt;   // the test hook withholds every load
                int j = 0;
                for (; j < nload; ++j) {
                    if (j > 0 && (j & 3) == 0) {
                        ecur = enext;
                        enext = load_entry((j / 4 + 1) * 32 + lane);
                    }
                    const int s = j % kT8Ring;
                    if (j >= kT8Ring) {
                        const bool ok = mbar_wait_bounded(code_free(s), static_cast<uint32_t>(((j / kT8Ring) - 1) & 1));
                        if (!__all_sync(kFull, ok)) {
                            timed_out = true;
                            break;
                        }
                    }
                    const int32_t e = __shfl_sync(kFull, ecur, (j & 3) * kTcBlocks + (lane & 7));
                    const int blk = bbase + j * kTcBlocks + lane;
                    const bool in = lane < kTcBlocks && blk < blk_end;
                    const bool v = in && e >= 0 && static_cast<int64_t>(e) < p.N;
                    if (in && !v) atomicOr(p.err, KVC_EBIT_BAD_BLOCK);
                    const uint32_t mask = __ballot_sync(kFull, v) & 0xFFu;
                    if (lane == 0) {
                        vmask_sh[s] = mask;   // for the converters; published by the arrive below
                        if (mask == 0u) mbar_arrive(code_full(s));
                        else
                            mbar_arrive_expect_tx(code_full(s),
                                                  static_cast<uint32_t>(__popc(mask)) * (2u * kBS * 128u));
                    }
                    __syncwarp();
                    if (v)
                        tma_load_2d(sbase + s * kT8CodeSlot + lane * (2 * kBS * 128), &tmap, code_full(s), 0,
                                    static_cast<int32_t>(((row_layer + e) * p.H_KV + h) * (2 * kBS)));
                }
                if (lane == 0)   // before the CTA exits: the last copies landed and their slots released
                    for (int jj = max(0, j - kT8Ring); jj < j; ++jj) {
                        (void)mbar_wait_bounded(code_full(jj % kT8Ring), static_cast<uint32_t>((jj / kT8Ring) & 1),
                                                100000000ull);
                        (void)mbar_wait_bounded(code_free(jj % kT8Ring), static_cast<uint32_t>((jj / kT8Ring) & 1),
                                                100000000ull);
                    }
                __syncwarp();
            } else if (warp == 5) {
                // ------------------------------------------------------------ MMA issuer
                constexpr uint32_t idesc_qk = tc_idesc_f16(128, G, false, false, false);
                constexpr uint32_t idesc_pv = tc_idesc_f16(128, 64, false, true, true);
                auto ready = [&](uint32_t bar, uint32_t parity) {   // lane 0 tests (never blocks), the warp agrees
                    const uint32_t r = lane == 0 ? (mbar_test_wait(bar, parity) ? 1u : 0u) : 0u;
                    return __shfl_sync(kFull, r, 0) != 0u;
                };
                const uint64_t desc_q = tc_smem_desc(sbase + kT8Q, 16, 1024, kSwizzle128B);
                bool q_ready = false;
                int jq = 0, jp = 0;
                uint64_t idle_since = 0;
                uint32_t idle = 0;
                while (jp < nt) {
                    bool progressed = false;
                    if (jp < jq && ready(pvready_bar(jp & 1), static_cast<uint32_t>((jp >> 1) & 1))) {
                        tc_fence_after();
                        const uint64_t desc_v = tc_smem_desc(sbase + kT8VF + (jp & 1) * kTcSlot, kTcBand, 1024,
                                                             kSwizzle128B);
                        const uint64_t desc_p = tc_smem_desc(sbase + kT8P + (jp & 1) * (kTcTok * 128), kTcBand, 1024,
                                                             kSwizzle128B);
#pragma unroll
                        for (int kk = 0; kk < kTcTok / 16; ++kk)   // 16 tokens (2048 bytes of rows) per MMA
                            tc_mma_f16_warp(tm_o, tc_desc_advance(desc_v, kk * 2048),
                                            tc_desc_advance(desc_p, kk * 2048),
                                            idesc_pv, (jp > 0 || kk > 0) ? 1u : 0u);
                        tc_commit_warp(pvdone_bar(jp & 1));
                        __syncwarp();
                        ++jp;
                        progressed = true;
                    }
                    if (!q_ready) q_ready = ready(qready_bar, 0u);
                    if (jq < nt && q_ready && ready(kf_full(jq & 1), static_cast<uint32_t>((jq >> 1) & 1)) &&
                        (jq < 2 || ready(sfree_bar(jq & 1), static_cast<uint32_t>(((jq - 2) >> 1) & 1)))) {
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)   // 16 channels (8 TMEM columns of A) per MMA
                            tc_mma_f16_tmem_a_warp(tmem + (jq & 1) * 32, tm_k + (jq & 1) * 64 + kk * 8,
                                                   tc_desc_advance(desc_q, (kk >> 2) * (32 * 128) + (kk & 3) * 32),
                                                   idesc_qk, kk > 0 ? 1u : 0u);
                        tc_commit_warp(sfull_bar(jq & 1));
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
                // before the CTA exits: every MMA issued has completed (they complete in order; immediate
                // unless a wait expired)
                if (lane == 0 && jp > 0)
                    (void)mbar_wait_bounded(pvdone_bar((jp - 1) & 1), static_cast<uint32_t>(((jp - 1) >> 1) & 1),
                                            100000000ull);
                if (lane == 0 && jq > 0)
                    (void)mbar_wait_bounded(sfull_bar((jq - 1) & 1), static_cast<uint32_t>(((jq - 1) >> 1) & 1),
                                            100000000ull);
                __syncwarp();
            } else {
                // ------------------------------------------------------------ value converters (64 positions each)
                const int half = warp - 6;
                int j = 0;
                for (; j < nt; ++j) {
                    const int s = j % kT8Ring, vb = j & 1;
                    bool ok = mbar_wait_bounded(code_full(s), static_cast<uint32_t>((j / kT8Ring) & 1));
                    // the f16 value tile is free once the value MMA that read it two tiles ago has completed
                    if (j >= 2) ok = ok && mbar_wait_bounded(pvdone_bar(vb), static_cast<uint32_t>(((j - 2) >> 1) & 1));
                    if (!__all_sync(kFull, ok)) {
                        timed_out = true;
                        break;
                    }
                    const uint32_t mask = vmask_sh[s];
                    const uint32_t code = sbase + s * kT8CodeSlot;
                    const int tok0 = blk0 * kBS + j * kTcTok;
                    // item (lane, k): token t = 64 half + lane / 8 + 4 k, 16-channel chunk c = lane mod 8
                    // (channels 16 c .. 16 c + 15: band c / 4, 16-byte chunks 2 (c mod 4) and + 1 of the f16
                    // row).  The upper band's lanes store their two chunks in the other order, so that each
                    // store of 8 lanes covers the 8 chunk positions of a row once (no bank conflict).
                    const int c = lane & 7, up = c >> 2;
                    const uint32_t band = sbase + kT8VF + vb * kTcSlot + up * kTcBand;
                    auto put = [&](int t, const uint4 &w, bool use) {
                        uint32_t f[8];
                        e4m3x16_to_f16(w, f);
                        uint4 out0 = make_uint4(f[0], f[1], f[2], f[3]), out1 = make_uint4(f[4], f[5], f[6], f[7]);
                        if (!use) out0 = out1 = make_uint4(0u, 0u, 0u, 0u);   // rows that must not count
                        sts128(band + sw128(t, 2 * (c & 3) + up), up ? out1 : out0);
                        sts128(band + sw128(t, 2 * (c & 3) + 1 - up), up ? out0 : out1);
                    };
#pragma unroll
                    for (int kk = 0; kk < 16; kk += 8) {   // 8 loads in flight, then their conversions
                        uint4 w[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int t = 64 * half + (lane >> 3) + 4 * (kk + k);
                            const int row = (t >> 4) * 2 * kBS + kBS + (t & 15);   // value row of the code slot
                            w[k] = lds128(code + row * 128 + ((c ^ (row & 7)) << 4));
                        }
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int t = 64 * half + (lane >> 3) + 4 * (kk + k);
                            put(t, w[k], ((mask >> (t >> 4)) & 1u) && tok0 + t < len);
                        }
                    }
                    // fused append: the step's own value row, quantised with the layer's scales, into the pool
                    // (its block is the sequence's last) and over its stale row of the tile, by the lanes that
                    // wrote that row above
                    const int t = app - tok0;
                    if (t >= 64 * half && t < 64 * half + 64 && ((mask >> (t >> 4)) & 1u) && (lane >> 3) == (t & 3)) {
                        const uint16_t *src = p.v_new + (static_cast<size_t>(b) * p.H_KV + h) * D + c * 16;
                        uint32_t qw[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) qw[i] = quantize4_e4m3(src + 4 * i, s_v + c * 16 + 4 * i);
                        const uint4 w = make_uint4(qw[0], qw[1], qw[2], qw[3]);
                        const int64_t el = ((((row_layer + app_phys) * p.H_KV + h) * 2 + 1) * kBS + app % kBS) * D;
                        *reinterpret_cast<uint4 *>(p.pool + el + c * 16) = w;
                        put(t, w, true);
                    }
                    fence_proxy_async_smem();   // before the tensor cores read the tile
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(pvready_bar(vb));
                        mbar_arrive(code_free(s));
                    }
                }
                // before the CTA exits: the value MMAs of the last two tiles released their tiles (immediate
                // unless a wait expired)
                if (lane == 0)
                    for (int jj = max(0, j - 2); jj < j; ++jj)
                        (void)mbar_wait_bounded(pvdone_bar(jj & 1), static_cast<uint32_t>((jj >> 1) & 1), 100000000ull);
                __syncwarp();
            }
        } else if (warp >= 8) {
            regs_down_128();
            // ------------------------------------------------------------ key wideners (thread = token)
            const int tq = 32 * (warp - 8) + lane;           // token of the tile; TMEM lane quarter warp mod 4
            const uint32_t lane_off = static_cast<uint32_t>(32 * (warp - 8)) << 16;
            int jj = 0;
            for (; jj < nt; ++jj) {
                const int s = jj % kT8Ring;
                // the codes have landed, and K[jj mod 2] is free once the score MMA of tile jj - 2 completed
                bool ok = mbar_wait_bounded(code_full(s), static_cast<uint32_t>((jj / kT8Ring) & 1));
                if (jj >= 2)
                    ok = ok && mbar_wait_bounded(sfull_bar(jj & 1), static_cast<uint32_t>(((jj - 2) >> 1) & 1));
                if (!__all_sync(kFull, ok)) {   // warp-uniform: the TMEM store below is warp-wide
                    timed_out = true;
                    break;
                }
                tc_fence_after();
                const uint32_t mask = vmask_sh[s];
                const int tok0 = blk0 * kBS + jj * kTcTok;
                const bool use = ((mask >> (tq >> 4)) & 1u) && tok0 + tq < len;
                const uint32_t code = sbase + s * kT8CodeSlot;
                const int row = (tq >> 4) * 2 * kBS + (tq & 15);   // key row of the code slot
                // the step's own key row, if this warp holds it: lane l quantises channels 4 l .. 4 l + 3
                const int ta = app - tok0;
                const bool mine = ta >= 32 * (warp - 8) && ta < 32 * (warp - 8) + 32 && ((mask >> (ta >> 4)) & 1u);
                uint32_t alo = 0u, ahi = 0u;
                if (mine) {
                    const uint32_t qw =
                        quantize4_e4m3(p.k_new + (static_cast<size_t>(b) * p.H_KV + h) * D + 4 * lane, s_k + 4 * lane);
                    const int64_t el = ((((row_layer + app_phys) * p.H_KV + h) * 2) * kBS + app % kBS) * D;
                    *reinterpret_cast<uint32_t *>(p.pool + el + 4 * lane) = qw;
                    e4m3x4_to_f16x2x2(qw, alo, ahi);
                }
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {   // channels 64 hf .. 64 hf + 63: columns 32 hf .. 32 hf + 31
                    uint4 w[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) w[c] = lds128(code + row * 128 + (((4 * hf + c) ^ (row & 7)) << 4));
                    uint32_t kw[32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) e4m3x16_to_f16(w[c], kw + 8 * c);
                    if (!use) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) kw[i] = 0u;
                    }
                    if (mine) {   // word g (channels 2 g, 2 g + 1) of the own row is lane g / 2's low or high word
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int g = 32 * hf + i;
                            const uint32_t v = __shfl_sync(kFull, (g & 1) ? ahi : alo, g >> 1);
                            if (tq == ta) kw[i] = v;
                        }
                    }
                    tmem_st32(tm_k + (jj & 1) * 64 + 32 * hf + lane_off, kw);
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(kf_full(jj & 1));
                __syncwarp();
                if (lane == 0) mbar_arrive(code_free(s));   // this warp's key rows are read
            }
        } else {
            regs_up_240();
            // ------------------------------------------------------------ softmax (128 threads)
            const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
            bool late = false;   // a wait that expired outside a vote: reported at the next vote
            float lp[G];
#pragma unroll
            for (int i = 0; i < G; ++i) lp[i] = 0.f;
            auto load_refs = [&](float (&mv)[G]) {
#pragma unroll
                for (int i = 0; i < G; i += 4) {
                    const float4 t = *reinterpret_cast<const float4 *>(msh + i);
                    mv[i] = t.x;
                    mv[i + 1] = t.y;
                    mv[i + 2] = t.z;
                    mv[i + 3] = t.w;
                }
            };
            int32_t ecur = load_entry(lane), enext = load_entry(32 + lane);
            int j = 0;
            for (; j < nt; ++j) {
                if (j > 0 && (j & 3) == 0) {
                    ecur = enext;
                    enext = load_entry((j / 4 + 1) * 32 + lane);
                }
                const int32_t e_tok = __shfl_sync(kFull, ecur, (j & 3) * kTcBlocks + 2 * warp + (lane >> 4));
                const int sb = j & 1;
                const bool ok1 = mbar_wait_bounded(sfull_bar(sb), static_cast<uint32_t>((j >> 1) & 1));
                tc_fence_after();
                uint32_t r[32];
                tmem_ld32(tmem + sb * 32 + lane_off, r);
                tmem_ld_wait(r);
                tc_fence_before();
                mbar_arrive(sfree_bar(sb));

                const int tok0 = blk0 * kBS + j * kTcTok;
                const int tok = tok0 + tid;
                const bool valid = tok < len && e_tok >= 0 && static_cast<int64_t>(e_tok) < p.N;
                float d[G];
                float dmax = -INFINITY;
                if (valid) {
                    load_refs(d);
#pragma unroll
                    for (int i = 0; i < G; ++i) {
                        d[i] = fmaf(__uint_as_float(r[i]), p.scale_log2, -d[i]);
                        dmax = fmaxf(dmax, d[i]);
                    }
                }
                // one CTA-wide vote per tile: a wait that expired, or a reference to move (which waits for
                // the previous value MMA before O^T is rescaled)
                bool pv_waited = false;
                if (softmax_any(!ok1 || late || dmax > kRescaleSlack)) {
                    const bool ok2 = j == 0 || mbar_wait_bounded(pvdone_bar((j - 1) & 1),
                                                                 static_cast<uint32_t>(((j - 1) >> 1) & 1));
                    if (!softmax_all(ok1 && ok2 && !late)) {
                        timed_out = true;
                        break;
                    }
                    tc_fence_after();
                    pv_waited = true;
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = valid ? __uint_as_float(r[i]) * p.scale_log2 : -INFINITY;
                    red[warp * 32 + lane] = warp_transpose_reduce<true>(v, lane);
                    softmax_sync();
                    if (warp == 0) {
                        const float M = fmaxf(fmaxf(red[lane], red[32 + lane]), fmaxf(red[64 + lane], red[96 + lane]));
                        const float mo = msh[lane];
                        const float mn = M > mo + kRescaleSlack ? M : mo;
                        msh[lane] = mn;
                        ash[lane] = mn == mo ? 1.f : fast_exp2(mo - mn);
                    }
                    softmax_sync();
                    bool moved = false;
#pragma unroll
                    for (int i = 0; i < G; ++i) {
                        const float a = ash[i];
                        lp[i] *= a;
                        moved |= a != 1.f;
                    }
                    if (moved && j > 0) {
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            uint32_t o[32];
                            tmem_ld32(tm_o + half * 32 + lane_off, o);
                            tmem_ld_wait(o);
#pragma unroll
                            for (int i = 0; i < G; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * ash[i]);
                            tmem_st32(tm_o + half * 32 + lane_off, o);
                        }
                        tmem_st_wait();
                    }
                    if (valid) {
                        load_refs(d);
#pragma unroll
                        for (int i = 0; i < G; ++i) d[i] = fmaf(__uint_as_float(r[i]), p.scale_log2, -d[i]);
                    }
                }
                // P^T[j mod 2] is free once the value MMA of tile j - 2 has completed (implied by j - 1's)
                if (!pv_waited && j >= 2)
                    late |= !mbar_wait_bounded(pvdone_bar(sb), static_cast<uint32_t>(((j - 2) >> 1) & 1));
                // this token's weights into row `tid` of P^T[j mod 2], 8 heads (one 16-byte chunk) at a time:
                // f16 high parts in columns 0..31, the f16 of the remainders in 32..63
                const uint32_t pst = sbase + kT8P + sb * (kTcTok * 128);
#pragma unroll
                for (int c = 0; c < G / 8; ++c) {
                    uint32_t pk[4] = {0u, 0u, 0u, 0u}, pl[4] = {0u, 0u, 0u, 0u};
                    if (valid) {
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const int i = 8 * c + 2 * k;
                            const float p0 = fast_exp2(d[i]), p1 = fast_exp2(d[i + 1]);
                            lp[i] += p0;
                            lp[i + 1] += p1;
                            pk[k] = pack_f16(p0, p1);
                            const __half2 hk = *reinterpret_cast<const __half2 *>(&pk[k]);
                            pl[k] = pack_f16(p0 - __low2float(hk), p1 - __high2float(hk));
                        }
                    }
                    sts128(pst + sw128(tid, c), make_uint4(pk[0], pk[1], pk[2], pk[3]));
                    sts128(pst + sw128(tid, c + 4), make_uint4(pl[0], pl[1], pl[2], pl[3]));
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(pvready_bar(sb));
            }

            // ---- epilogue: O^T (thread = channel) times s_V, the per-head sums, output or partial
            bool ok = !timed_out && !late &&
                      mbar_wait_bounded(pvdone_bar((nt - 1) & 1), static_cast<uint32_t>(((nt - 1) >> 1) & 1));
            ok = softmax_all(ok);
            if (!ok) {
                timed_out = true;
            } else {
                tc_fence_after();
                uint32_t o[32], olo[32];
                tmem_ld32(tm_o + lane_off, o);
                tmem_ld_wait(o);
                tmem_ld32(tm_o + 32 + lane_off, olo);
                tmem_ld_wait(olo);
                const float sv = __ldg(s_v + tid);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    o[i] = __float_as_uint((__uint_as_float(o[i]) + __uint_as_float(olo[i])) * sv);
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = lp[i];
                red[warp * 32 + lane] = warp_transpose_reduce<false>(v, lane);
                softmax_sync();
                if (warp == 0) lsh[lane] = (red[lane] + red[32 + lane]) + (red[64 + lane] + red[96 + lane]);
                softmax_sync();
                const size_t row0 = static_cast<size_t>(b) * p.H_Q + hq0;
                if (ns == 1) {
#pragma unroll
                    for (int i = 0; i < G; ++i) p.out[(row0 + i) * D + tid] = __uint_as_float(o[i]) / lsh[i];
                    if (p.lse && tid < G) p.lse[row0 + tid] = (msh[tid] + log2f(lsh[tid])) * kLn2;
                } else {
#pragma unroll
                    for (int i = 0; i < G; ++i)
                        p.part_o[((row0 + i) * p.max_splits + split) * D + tid] = __uint_as_float(o[i]);
                    if (tid < G) p.part_ml[(row0 + tid) * p.max_splits + split] = make_float2(msh[tid], lsh[tid]);
                }
            }
        }
        if (timed_out && lane == 0) atomicOr(p.err, KVC_EBIT_TIMEOUT);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kT8Cols);
    }
}

// grid (split, KV head, sequence), 384 threads
template <int G>
__global__ void __launch_bounds__(kT8Threads, 1) decode_tc8_kernel(const __grid_constant__ CUtensorMap tmap,
                                                                   const DecodeParams p)
{
    allow_dependent_launch();
    decode_tc8_cta<G>(tmap, p, blockIdx.x, blockIdx.y, blockIdx.z);
}

}  // namespace kvc
