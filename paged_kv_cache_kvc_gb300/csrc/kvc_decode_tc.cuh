// Paged decode attention for large query groups (MQA: 32 query heads per KV
// head) on the fifth-generation tensor cores, with scores and outputs in
// tensor memory (TMEM).
//
// What it computes is the split kernel's ("KV cache: Generation state,
// latency, and allocation" 21.1 and 21.5; the xf_kv_cache page: GQA / MQA
// head sharing): for sequence b, KV head h and its G query heads,
// softmax(scale * q K^T) V over the n = lens[b] positions the table maps.
//
// Why a second kernel: with G = 32 query columns a warp-level mma kernel
// holds 32 x 128 fp32 accumulators per thread, so few warps fit an SM and
// dependent mma chains leave HBM idle.  Here one thread issues 128-token MMAs
// whose accumulators live in TMEM, and the registers hold one token's scores.
//
// CTA = one split of (b, h); 224 threads in four roles:
//   warps 4, 6  TMA producers, one for keys and one for values: per 128-token
//               tile, the 8 blocks' key rows (or value rows) as 16-row boxes
//               (128-byte swizzle) into a ring of 3 slots of 32 KiB
//               ([2 bands][128 tokens][128 B]).  A key slot is released as soon
//               as the tile's score MMA has completed and a value slot when its
//               value MMA has: keys run ahead, values are fetched for later.
//   warp 5      MMA issuer (one lane):
//                 S^T[128 tok x G]  = K[128 x 128] . Q^T     (K-major A and B)
//                 O^T[128 ch x 64] += V^T[128 x 128] . P^T    (MN-major A and B)
//               S double-buffered in TMEM, O^T in TMEM.  P^T's 64 columns (one
//               128-byte swizzle atom) hold each weight as a bf16 high part
//               (columns 0..31) and the bf16 of its remainder (32..63), so O^T
//               accumulates the two halves apart and the epilogue adds them:
//               about 16 bits of every weight reach the value mixture.  It also
//               zeroes value rows of positions that must not count (0 * NaN is
//               NaN) and, for the fused step, writes the appended row.
//   warps 0..3  softmax, thread t = token t of the tile (TMEM lane t):
//               x = scale * s (log2 units), p = 2^(x - m_ref) with a per-head
//               reference max m_ref that moves only when some score exceeds it
//               by more than 8 (then O^T and the partial sums are rescaled by
//               2^(m_old - m_new); conditional rescaling as in FlashAttention-4).
//               Whether any head must move is one CTA-wide vote (bar.red.or);
//               only then are per-head maxima reduced across the 128 threads.
//               P^T row t (high and low bf16 parts) goes to shared memory.
// Epilogue: O^T from TMEM (thread = channel), per-head sums reduced across
// threads, then the final output (one split) or a split partial for the merge.
#pragma once
#include "kvc_decode.cuh"
#include "kvc_tc.cuh"

namespace kvc {

constexpr int kTcTok = 128;                         // tokens per tile: the MMA's M
constexpr int kTcBlocks = kTcTok / kBS;             // 8 blocks per tile
constexpr int kTcThreads = 224;
constexpr int kTcRing = 3;
constexpr int kTcBand = kTcTok * 128;               // one 128-byte column band of 128 rows
constexpr int kTcSlot = 2 * kTcBand;                // the keys (or the values) of a tile: 2 bands, d_h 128 bf16
constexpr int kTcV = kTcRing * kTcSlot;             // key slots first, then value slots
constexpr int kTcQ = 2 * kTcRing * kTcSlot;         // Q: 2 bands x 32 head rows x 128 B
constexpr int kTcP = kTcQ + 2 * 32 * 128;           // P^T: 128 token rows x 64 bf16 heads
constexpr int kTcBars = kTcP + kTcTok * 128;
// barriers: kfull[R], kfree[R], vfull[R], vfree[R], s_full[2], s_free[2], p_full, pv_done, q_ready
constexpr int kTcNumBars = 4 * kTcRing + 7;
// float [4][32] reductions, then msh[32], ash[32], lsh[32] (16-byte aligned: read as float4)
constexpr int kTcRed = kTcBars + ((kTcNumBars * 8 + 15) & ~15);
constexpr int kTcTmemSlot = kTcRed + (4 * 32 + 3 * 32) * 4;
constexpr int kTcSmem = 1024 + kTcTmemSlot + 16;
constexpr uint32_t kTcCols = 128;   // TMEM: S[0] 0..31, S[1] 32..63, O^T 64..127 (high part, then low part)

// Named barriers of the 128 softmax threads (0 is __syncthreads).
__device__ __forceinline__ bool softmax_all(bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, 1, 128, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"(v ? 1u : 0u)
                 : "memory");
    return r != 0;
}

__device__ __forceinline__ bool softmax_any(bool v)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, 128, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r)
                 : "r"(v ? 1u : 0u)
                 : "memory");
    return r != 0;
}

__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// Lane l ends with the reduction over the warp's 32 lanes of v[l]: each step
// halves the values a lane keeps, exchanging the other half with its partner.
template <bool MAX>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[32], int lane)
{
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) {
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < s; ++i) {
            const float send = upper ? v[i] : v[i + s];
            const float keep = upper ? v[i + s] : v[i];
            const float got = __shfl_xor_sync(kFull, send, s);
            v[i] = MAX ? fmaxf(keep, got) : keep + got;
        }
    }
    return v[0];
}

// One split of unit (b, h), G query heads (G = 32).
template <int G>
__device__ __forceinline__ void decode_tc_cta(const CUtensorMap &tmap16, const DecodeParams &p, const int split,
                                              const int h, const int b)
{
    static_assert(G == 32, "the TMEM score buffers and the head reductions are laid out for 32 heads");
    constexpr int D = 128;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hq0 = h * p.g;

    const uint32_t sbase = smem_u32(smem);
    const uint32_t bars = sbase + kTcBars;
    // kv = 0: key slots, 1: value slots
    auto full_bar = [&](int kv, int s) { return bars + 8u * (2 * kv * kTcRing + s); };
    auto free_bar = [&](int kv, int s) { return bars + 8u * (2 * kv * kTcRing + kTcRing + s); };
    auto sfull_bar = [&](int sb) { return bars + 8u * (4 * kTcRing + sb); };
    auto sfree_bar = [&](int sb) { return bars + 8u * (4 * kTcRing + 2 + sb); };
    const uint32_t pfull_bar = bars + 8u * (4 * kTcRing + 4);
    const uint32_t pvdone_bar = bars + 8u * (4 * kTcRing + 5);
    const uint32_t qready_bar = bars + 8u * (4 * kTcRing + 6);
    float *red = reinterpret_cast<float *>(smem + kTcRed);   // [4][32]
    float *msh = red + 128, *ash = msh + 32, *lsh = ash + 32;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kTcTmemSlot);

    // ---- set-up, before any global memory access: barriers, TMEM, reference maxima
    if (tid == 0) {
        for (int kv = 0; kv < 2; ++kv)
            for (int s = 0; s < kTcRing; ++s) {
                mbar_init(full_bar(kv, s), 1);
                mbar_init(free_bar(kv, s), 1);
            }
        for (int sb = 0; sb < 2; ++sb) {
            mbar_init(sfull_bar(sb), 1);
            mbar_init(sfree_bar(sb), 128);
        }
        mbar_init(pfull_bar, 128);
        mbar_init(pvdone_bar, 1);
        mbar_init(qready_bar, 128);
        fence_barrier_init();
        prefetch_tensormap(&tmap16);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), kTcCols);
        tmem_relinquish();
    }
    if (tid < 32) msh[tid] = -INFINITY;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // While the kernel before it drains: a speculative L2 prefetch of the split's first 3
    // tiles, from the lengths and table as they stand now (they may still change; nothing
    // here is used but as a cache hint, and everything below the wait reads them again).
    if (tid < kTcRing * kTcBlocks && p.lens && p.pool) {
        const int len_s = p.lens[b] + (p.k_new ? 1 : 0);
        const int blk = split * p.chunk + tid;
        if (blk < p.max_blocks && blk * kBS < len_s) {
            const int32_t e = p.bt[static_cast<int64_t>(b) * p.bt_stride + blk];
            if (e >= 0 && static_cast<int64_t>(e) < p.N)
                prefetch_l2_bulk(p.pool + ((static_cast<int64_t>(p.layer) * p.N + e) * p.H_KV + h) * (2 * kBS * D * 2),
                                 2 * kBS * D * 2);
        }
    }
    // Launched as a programmatic dependent of the kernel before it on the stream: the set-up
    // above overlaps that kernel's tail, and this wait (a no-op in an ordinary launch) holds
    // the CTA until that kernel has finished and its writes are visible.  Everything below
    // reads or writes global memory.
    grid_dependency_wait();

    int len = seq_len(p, b);
    if (len < 0 || static_cast<int64_t>(len) > static_cast<int64_t>(p.max_blocks) * kBS) {
        if (split == 0 && tid == 0) atomicOr(p.err, KVC_EBIT_RANGE);
        len = 0;
    }
    const int nblk = (len + kBS - 1) / kBS;
    if (nblk == 0 && split == 0) {   // empty sequence: zero output, lse = -inf
        for (int i = tid; i < G * D; i += kTcThreads) p.out[(static_cast<size_t>(b) * p.H_Q + hq0) * D + i] = 0.f;
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

        if (tid < 128) {   // q rows (K-major B operand of the score MMA), while the first keys are in flight
            for (int i = tid; i < G * 16; i += 128) {   // row hh, 16-byte chunk c of 16
                const int hh = i >> 4, c = i & 15;
                const size_t qi = (static_cast<size_t>(b) * p.H_Q + hq0 + hh) * D + c * 8;
                const uint4 v = *reinterpret_cast<const uint4 *>(p.q + qi);
                sts128(sbase + kTcQ + (c >> 3) * (32 * 128) + sw128(hh, c & 7), v);
            }
            fence_proxy_async_smem();
            mbar_arrive(qready_bar);
        }
        const uint32_t tm_o = tmem + 64;

        bool timed_out = false;
        // table entries of the CTA's blocks, 32 (4 tiles) at a time in registers, one window ahead:
        // lane l holds block 32 w + l of window w
        const int bbase = blk0;
        auto load_entry = [&](int rel) -> int32_t { return bbase + rel < blk_end ? __ldg(bt_row + bbase + rel) : -1; };

        if (warp == 4 || warp == 6) {
            // ------------------------------------------------------------ TMA producers (4: keys, 6: values)
            const int kv = warp == 6 ? 1 : 0;
            int32_t ecur = load_entry(lane), enext = load_entry(32 + lane);
            const int nload = p.stall_loads ? 0 : nt;   // the test hook withholds every load
            int j = 0;
            for (; j < nload; ++j) {
                if (j > 0 && (j & 3) == 0) {
                    ecur = enext;
                    enext = load_entry((j / 4 + 1) * 32 + lane);
                }
                const int s = j % kTcRing;
                if (j >= kTcRing) {
                    const bool ok = mbar_wait_bounded(free_bar(kv, s), static_cast<uint32_t>(((j / kTcRing) - 1) & 1));
                    if (!__all_sync(kFull, ok)) {
                        timed_out = true;
                        break;
                    }
                }
                const int32_t e = __shfl_sync(kFull, ecur, (j & 3) * kTcBlocks + (lane & 7));
                const int blk = bbase + j * kTcBlocks + lane;
                const bool in = lane < kTcBlocks && blk < blk_end;
                const bool v = in && e >= 0 && static_cast<int64_t>(e) < p.N;
                if (kv == 0 && in && !v) atomicOr(p.err, KVC_EBIT_BAD_BLOCK);
                const uint32_t mask = __ballot_sync(kFull, v);
                if (lane == 0) {
                    if (mask == 0u) mbar_arrive(full_bar(kv, s));
                    else
                        mbar_arrive_expect_tx(full_bar(kv, s), static_cast<uint32_t>(__popc(mask)) * 2u * (kBS * 128u));
                }
                __syncwarp();
                // one box per lane, all in one instruction: lane = (band, block); every lane
                // already holds the entry of block lane mod 8
                if (lane < 2 * kTcBlocks && ((mask >> (lane & 7)) & 1u)) {
                    const int32_t y = static_cast<int32_t>(((row_layer + e) * p.H_KV + h) * (2 * kBS) + kv * kBS);
                    tma_load_2d(sbase + kv * kTcV + s * kTcSlot + (lane >> 3) * kTcBand + (lane & 7) * (kBS * 128),
                                &tmap16, full_bar(kv, s), (lane >> 3) * 64, y);
                }
            }
            // before the CTA exits: the copies of the last slots have landed and their releases
            // (tcgen05 commits, which arrive asynchronously) are in; both are immediate unless a
            // wait somewhere expired
            if (lane == 0)
                for (int jj = max(0, j - kTcRing); jj < j; ++jj) {
                    (void)mbar_wait_bounded(full_bar(kv, jj % kTcRing), static_cast<uint32_t>((jj / kTcRing) & 1),
                                            100000000ull);
                    (void)mbar_wait_bounded(free_bar(kv, jj % kTcRing), static_cast<uint32_t>((jj / kTcRing) & 1),
                                            100000000ull);
                }
            __syncwarp();
        } else if (warp == 5) {
            // ------------------------------------------------------------ MMA issuer
            // Issues whichever MMA is ready: the score MMA of tile jq once its keys have landed and
            // its score buffer is free (it releases the key slot), the value MMA of tile jp once its
            // weights are in shared memory and its values have landed (it releases the value slot).
            // Barriers are tested without blocking.
            constexpr uint32_t idesc_qk = tc_idesc_f16(128, G, true, false, false);
            constexpr uint32_t idesc_pv = tc_idesc_f16(128, 64, true, true, true);
            int32_t ecur = load_entry(lane), enext = load_entry(32 + lane);
            auto ready = [&](uint32_t bar, uint32_t parity) {   // lane 0 tests (never blocks), the warp agrees
                const uint32_t r = lane == 0 ? (mbar_test_wait(bar, parity) ? 1u : 0u) : 0u;
                return __shfl_sync(kFull, r, 0) != 0u;
            };
            const uint64_t desc_q = tc_smem_desc(sbase + kTcQ, 16, 1024, kSwizzle128B);
            const uint64_t desc_p = tc_smem_desc(sbase + kTcP, kTcBand, 1024, kSwizzle128B);
            // per tile in flight (3 at most between score and value MMA): its valid blocks, 8 bits each
            uint32_t vmasks = 0u;
            int32_t append_phys = -1;   // the block receiving the fused append (the sequence's last tile)
            bool q_ready = false;
            int jq = 0, jp = 0;
            uint64_t idle_since = 0;
            uint32_t idle = 0;
            while (jp < nt) {
                bool progressed = false;
                if (jp < jq && ready(pfull_bar, static_cast<uint32_t>(jp & 1)) &&
                    ready(full_bar(1, jp % kTcRing), static_cast<uint32_t>((jp / kTcRing) & 1))) {
                    const uint32_t vst = sbase + kTcV + (jp % kTcRing) * kTcSlot;
                    // positions that must contribute nothing: past the sequence end, or in a block whose
                    // table entry is bad; their value rows are zeroed (their weights are 0; 0 * NaN is not)
                    const int tok0 = blk0 * kBS + jp * kTcTok;
                    const uint32_t vmask = (vmasks >> (8 * (jp % kTcRing))) & 0xFFu;
                    bool fix = tok0 + kTcTok > len || vmask != 0xFFu;
                    if (fix) {
                        for (int i = lane; i < kTcTok * 16; i += 32) {
                            const int row = i >> 4, c = i & 15, tok = tok0 + row;
                            if (tok >= len || !(vmask >> (row >> 4) & 1u))
                                sts128_zero(vst + (c >> 3) * kTcBand + sw128(row, c & 7));
                        }
                    }
                    // fused append: the step's own value row, into the pool and into the slot
                    if (p.k_new && tok0 <= len - 1 && len - 1 < tok0 + kTcTok && append_phys >= 0) {
                        fix = true;
                        if (lane < 16) {
                            const int row = len - 1 - tok0, c = lane;
                            const uint4 val = *reinterpret_cast<const uint4 *>(
                                p.v_new + (static_cast<size_t>(b) * p.H_KV + h) * D + c * 8);
                            const int64_t el =
                                ((((row_layer + append_phys) * p.H_KV + h) * 2 + 1) * kBS + (row & 15)) * D + c * 8;
                            *reinterpret_cast<uint4 *>(p.pool + el * 2) = val;
                            sts128(vst + (c >> 3) * kTcBand + sw128(row, c & 7), val);
                        }
                    }
                    if (fix) fence_proxy_async_smem();   // zeros / the appended row, before the tensor cores read them
                    __syncwarp();
                    tc_fence_after();
                    {
                        const uint64_t a0 = tc_smem_desc(vst, kTcBand, 1024, kSwizzle128B);
#pragma unroll
                        for (int kk = 0; kk < kTcTok / 16; ++kk)   // 16 tokens (2048 bytes of rows) per MMA
                            tc_mma_f16_warp(tm_o, tc_desc_advance(a0, kk * 2048), tc_desc_advance(desc_p, kk * 2048),
                                            idesc_pv, (jp > 0 || kk > 0) ? 1u : 0u);
                        tc_commit_warp(free_bar(1, jp % kTcRing));
                        tc_commit_warp(pvdone_bar);
                    }
                    __syncwarp();
                    ++jp;
                    progressed = true;
                }
                if (!q_ready) q_ready = ready(qready_bar, 0u);
                if (jq < nt && jq < jp + kTcRing && q_ready &&
                    ready(full_bar(0, jq % kTcRing), static_cast<uint32_t>((jq / kTcRing) & 1)) &&
                    (jq < 2 || ready(sfree_bar(jq & 1), static_cast<uint32_t>(((jq - 2) >> 1) & 1)))) {
                    if (jq > 0 && (jq & 3) == 0) {
                        ecur = enext;
                        enext = load_entry((jq / 4 + 1) * 32 + lane);
                    }
                    const uint32_t kst = sbase + (jq % kTcRing) * kTcSlot;
                    const int tok0 = blk0 * kBS + jq * kTcTok;
                    const int32_t e = __shfl_sync(kFull, ecur, (jq & 3) * kTcBlocks + (lane & 7));
                    const bool bv =
                        bbase + jq * kTcBlocks + (lane & 7) < blk_end && e >= 0 && static_cast<int64_t>(e) < p.N;
                    const uint32_t vmask = __ballot_sync(kFull, bv) & 0xFFu;
                    vmasks = (vmasks & ~(0xFFu << (8 * (jq % kTcRing)))) | (vmask << (8 * (jq % kTcRing)));
                    // fused append: the step's own key row, into the pool and into the slot (its value row
                    // goes in at the value MMA)
                    bool wrote = false;
                    if (p.k_new && tok0 <= len - 1 && len - 1 < tok0 + kTcTok) {
                        const int row = len - 1 - tok0;
                        const int32_t phys = __shfl_sync(kFull, e, row >> 4);
                        if ((vmask >> (row >> 4)) & 1u) {
                            append_phys = phys;
                            wrote = true;
                            if (lane < 16) {
                                const int c = lane;
                                const uint4 val = *reinterpret_cast<const uint4 *>(
                                    p.k_new + (static_cast<size_t>(b) * p.H_KV + h) * D + c * 8);
                                const int64_t el =
                                    ((((row_layer + phys) * p.H_KV + h) * 2) * kBS + (row & 15)) * D + c * 8;
                                *reinterpret_cast<uint4 *>(p.pool + el * 2) = val;
                                sts128(kst + (c >> 3) * kTcBand + sw128(row, c & 7), val);
                            }
                        }
                    }
                    if (wrote) fence_proxy_async_smem();
                    __syncwarp();
                    tc_fence_after();
                    {
                        const uint64_t a0 = tc_smem_desc(kst, 16, 1024, kSwizzle128B);
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk)   // 16 channels (32 bytes) per MMA, 4 per 128-byte band
                            tc_mma_f16_warp(tmem + (jq & 1) * 32,
                                            tc_desc_advance(a0, (kk >> 2) * kTcBand + (kk & 3) * 32),
                                            tc_desc_advance(desc_q, (kk >> 2) * (32 * 128) + (kk & 3) * 32), idesc_qk,
                                            kk > 0 ? 1u : 0u);
                        tc_commit_warp(sfull_bar(jq & 1));
                        tc_commit_warp(free_bar(0, jq % kTcRing));
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
        } else {
            // ------------------------------------------------------------ softmax (128 threads)
            const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
            // this token's partial sums per head; the reference maxima (the same for every thread) are
            // read from their shared copy msh, which only the slow path below rewrites
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
            // table entries in the same register windows as the other roles (a warp's token of
            // tile j lies in block 8 j + 2 warp + lane / 16)
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

                const int tok = blk0 * kBS + j * kTcTok + tid;
                const bool valid = tok < len && e_tok >= 0 && static_cast<int64_t>(e_tok) < p.N;
                // d = scale s - m (log2 units) per head; a reference moves when some d exceeds the
                // slack (a reference of -inf: d = +inf).  Invalid positions weigh nothing.
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
                // P^T and O^T are free once the previous tile's value MMA has completed
                const bool ok2 = j == 0 || mbar_wait_bounded(pvdone_bar, static_cast<uint32_t>((j - 1) & 1));
                tc_fence_after();
                // one CTA-wide vote per tile: a wait that expired anywhere, or a reference to move
                if (softmax_any(!ok1 || !ok2 || dmax > kRescaleSlack)) {
                    if (!softmax_all(ok1 && ok2)) {
                        timed_out = true;
                        break;
                    }
                    // per-head tile maxima over the 128 tokens, new references and rescale factors
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
                    if (moved && j > 0) {   // O^T lane = channel, column = head (high, then low part)
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
                    if (valid) {   // against the new references (finite: this position's score is in the max)
                        load_refs(d);
#pragma unroll
                        for (int i = 0; i < G; ++i) d[i] = fmaf(__uint_as_float(r[i]), p.scale_log2, -d[i]);
                    }
                }
                // weights of this token for every head, into row `tid` of P^T, 8 heads (one 16-byte
                // chunk) at a time: bf16 high parts in columns 0..31, the bf16 of the remainders in 32..63
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
                            pk[k] = pack_bf16(p0, p1);
                            pl[k] = pack_bf16(p0 - bf16_lo(pk[k]), p1 - bf16_hi(pk[k]));
                        }
                    }
                    sts128(sbase + kTcP + sw128(tid, c), make_uint4(pk[0], pk[1], pk[2], pk[3]));
                    sts128(sbase + kTcP + sw128(tid, c + 4), make_uint4(pl[0], pl[1], pl[2], pl[3]));
                }
                fence_proxy_async_smem();
                tc_fence_before();
                mbar_arrive(pfull_bar);
            }

            // ---- epilogue: O^T (thread = channel), the per-head sums, output or split partial
            bool ok = !timed_out && mbar_wait_bounded(pvdone_bar, static_cast<uint32_t>((nt - 1) & 1));
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
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) + __uint_as_float(olo[i]));
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
        tmem_dealloc(tmem, kTcCols);
    }
}

// grid (split, KV head, sequence), 224 threads
template <int G>
__global__ void __launch_bounds__(kTcThreads, 1) decode_tc_kernel(const __grid_constant__ CUtensorMap tmap16,
                                                                  const DecodeParams p)
{
    allow_dependent_launch();
    decode_tc_cta<G>(tmap16, p, blockIdx.x, blockIdx.y, blockIdx.z);
}

// The tensor-memory decode kernel for a shape, or fn = nullptr (d_h 128 bf16 or e4m3 pools, 32-head groups).
DecodeKernel select_decode_tc(int D, int g, int dtype);
// The e4m3 form alone (kvc_decode_tc8.cu).
DecodeKernel select_decode_tc8(int D, int g);
// The same for a launch's parameters (decode steps only; fn = nullptr when KVC_TC=0).
DecodeKernel tc_kernel_for(const kvc_pool *pool, const DecodeParams &p);

}  // namespace kvc
