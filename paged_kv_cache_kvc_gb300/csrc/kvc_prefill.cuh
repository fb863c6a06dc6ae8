// Causal attention of a prefill chunk over a paged bf16 cache, queries on the
// tensor cores' M dimension ("KV cache: Generation state, latency, and
// allocation" 21.3: a chunked prefill keeps the earlier positions and adds the
// chunk's; the xf_kv_cache page, "End-to-end flow": the new tokens attend to
// the shared prefix through the row's table).
//
// Query i of the chunk sits at position q_start + i and reads positions
// 0 .. q_start + i.  A CTA (4 warps) takes KV head h and a tile of 64 / g
// consecutive chunk positions; warp w owns 16 consecutive positions of query
// head h * g + (w mod g), so the g heads that share a KV head share every
// staged key/value tile.  Per stage the CTA stages 64 keys (4 blocks of the
// row, one contiguous keys-then-values run per block and head, TMA with the
// 128-byte swizzle) in a ring of 3 stages; the last warp done with a stage
// refills it.  Each warp runs, on mma.sync m16n8k16 with fp32 accumulation:
//   S[16 pos x 64 keys]  = Q[16 x D] K^T          (Q fragments in registers)
//   online softmax per row (quad shuffles), causal mask on key > position
//   O[16 x D]           += P[16 x 64] V            (P re-packed from S in registers)
// Rows past the chunk end compute on zero queries and are not written.
#pragma once
#include "kvc_decode.cuh"

namespace kvc {

constexpr int kPrefillKeys = 64;   // keys per stage: 4 blocks
constexpr int kPrefillRing = 3;   // stages of the standalone kernel

template <int D, int RING = kPrefillRing>
struct PrefillCfg {
    static constexpr int BLK = 2 * kBS * D * 2;                 // one block-head of bf16 keys then values
    static constexpr int BLOCKS = kPrefillKeys / kBS;
    static constexpr int STAGE = BLOCKS * BLK;
    static constexpr int BANDS = D * 2 / 128;
    static constexpr int KSTEPS = D / 16;                       // QK k-steps
    static constexpr int NDIM = D / 8;                          // PV n-tiles
    static constexpr int SMEM = 1024 /* alignment slack */ + RING * STAGE + RING * 8 + 64;   // + masks, counts
};

// CTA (tile, h) of a prefill chunk: p.len_base = q_start, p.n_pos = n_q,
// p.ppu = 64 / g positions per tile, p.bt = the row's table, p.max_blocks >=
// the blocks holding positions < q_start + n_q.
template <int D, int RING = kPrefillRing>
__device__ __forceinline__ void prefill_cta(const CUtensorMap &tmap, const DecodeParams &p, const int tile,
                                            const int h)
{
    using C = PrefillCfg<D, RING>;
    constexpr int kPrefillRing = RING;   // this instance's stages
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kPrefillRing * C::STAGE);
    uint32_t *valid_mask = reinterpret_cast<uint32_t *>(bars + kPrefillRing);   // [ring] blocks staged per stage
    int *done_warps = reinterpret_cast<int *>(valid_mask + kPrefillRing);         // [ring] warps finished with it

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tg = lane & 3;
    const int g = p.g;
    const int hq = h * g + warp % g;                       // this warp's query head
    const int pos0 = tile * p.ppu + (warp / g) * 16;       // its first chunk position
    const int q_start = p.len_base, n_q = p.n_pos;
    const int total = q_start + n_q;                       // positions the chunk's row holds
    // keys this CTA needs: through its last real position
    const int n_keys = min(total, q_start + (tile + 1) * p.ppu);
    const int n_tiles = (n_keys + kPrefillKeys - 1) / kPrefillKeys;
    const int nblk = (n_keys + kBS - 1) / kBS;
    const int64_t row_layer = static_cast<int64_t>(p.layer) * p.N;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPrefillRing; ++s) {
            mbar_init(smem_u32(&bars[s]), 1);
            done_warps[s] = 0;
        }
        fence_barrier_init();
        prefetch_tensormap(&tmap);
    }
    __syncthreads();

    // stage tile jj (one thread): the row's blocks 4jj .. 4jj+3 that hold needed keys
    auto issue = [&](int jj) {
        const int s = jj % kPrefillRing;
        const uint32_t bar = smem_u32(&bars[s]);
        const uint32_t dst = smem_u32(smem + s * C::STAGE);
        uint32_t mask = 0, bytes = 0;
        int32_t phys[C::BLOCKS];
#pragma unroll
        for (int k = 0; k < C::BLOCKS; ++k) {
            const int blk = jj * C::BLOCKS + k;
            phys[k] = blk < nblk ? __ldg(p.bt + blk) : -1;
            if (blk < nblk && (phys[k] < 0 || static_cast<int64_t>(phys[k]) >= p.N)) atomicOr(p.err, KVC_EBIT_BAD_BLOCK);
            if (phys[k] >= 0 && static_cast<int64_t>(phys[k]) < p.N) {
                mask |= 1u << k;
                bytes += C::BLK;
            }
        }
        valid_mask[s] = mask;
        if (bytes == 0) {
            mbar_arrive(bar);
            return;
        }
        mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
        for (int k = 0; k < C::BLOCKS; ++k) {
            if (!(mask >> k & 1u)) continue;
            const int32_t y = static_cast<int32_t>(((row_layer + phys[k]) * p.H_KV + h) * (2 * kBS));
#pragma unroll
            for (int band = 0; band < C::BANDS; ++band)
                tma_load_2d(dst + k * C::BLK + band * 2 * kBS * 128, &tmap, bar, band * 64, y);
        }
    };
    if (threadIdx.x == 0)
        for (int jj = 0; jj < min(kPrefillRing, n_tiles); ++jj) issue(jj);
    __syncthreads();   // the first stages' masks are written

    // ---- query fragments (A operand: rows = positions pos0 + gq (+8), k = channel)
    uint32_t qf[C::KSTEPS][4];
    {
        const int r0 = pos0 + gq, r1 = pos0 + gq + 8;
        const uint16_t *q0 = p.q + (static_cast<size_t>(min(r0, n_q - 1)) * p.H_Q + hq) * D;
        const uint16_t *q1 = p.q + (static_cast<size_t>(min(r1, n_q - 1)) * p.H_Q + hq) * D;
#pragma unroll
        for (int kk = 0; kk < C::KSTEPS; ++kk) {
            const int c = 16 * kk + 2 * tg;
            qf[kk][0] = r0 < n_q ? *reinterpret_cast<const uint32_t *>(q0 + c) : 0u;
            qf[kk][1] = r1 < n_q ? *reinterpret_cast<const uint32_t *>(q1 + c) : 0u;
            qf[kk][2] = r0 < n_q ? *reinterpret_cast<const uint32_t *>(q0 + c + 8) : 0u;
            qf[kk][3] = r1 < n_q ? *reinterpret_cast<const uint32_t *>(q1 + c + 8) : 0u;
        }
    }
    const int vis0 = q_start + pos0 + gq + 1, vis1 = vis0 + 8;   // keys visible to this thread's two rows

    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    float oacc[C::NDIM][4];
#pragma unroll
    for (int nd = 0; nd < C::NDIM; ++nd) oacc[nd][0] = oacc[nd][1] = oacc[nd][2] = oacc[nd][3] = 0.f;

    // wait (bounded) for tile jj's stage; zero the value rows that must read as zero (their
    // weights are 0, but 0 * NaN is not): blocks not staged, and slots past the row's end.
    // Every warp zeroes them for itself (the same zeros; the stage's copies have landed).
    auto acquire = [&](int jj, uint32_t &st, uint32_t &mask) -> bool {
        const int s = jj % kPrefillRing;
        const bool ok = mbar_wait_bounded(smem_u32(&bars[s]), static_cast<uint32_t>((jj / kPrefillRing) & 1));
        if (!__all_sync(kFull, ok)) return false;
        st = smem_u32(smem + s * C::STAGE);
        mask = valid_mask[s];
        const int key0 = jj * kPrefillKeys;
        if (mask != (1u << C::BLOCKS) - 1u || key0 + kPrefillKeys > total) {
            for (int i = lane; i < C::BLOCKS * kBS * C::BANDS * 8; i += 32) {
                const int k = i / (kBS * C::BANDS * 8), rem = i - k * (kBS * C::BANDS * 8);
                const int slot = rem / (C::BANDS * 8), ch = rem - slot * (C::BANDS * 8);
                const bool dead = !(mask >> k & 1u) || key0 + k * kBS + slot >= total;
                if (dead) sts128_zero(st + k * C::BLK + swz(kBS + slot, ch));
            }
            __syncwarp();
        }
        return true;
    };

    // S = Q K^T over a stage's 64 keys (8 n-tiles of 8 keys)
    auto qk = [&](uint32_t st, float (&sc)[8][4]) {
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
            const int key = nt * 8 + (lane & 7);   // this lane's ldmatrix row
            const uint32_t krow = st + (key >> 4) * C::BLK;
#pragma unroll
            for (int kk = 0; kk < C::KSTEPS; kk += 2) {
                uint32_t b[4];
                ldsm_x4(b, krow + swz(key & 15, 2 * kk + (lane >> 3)));
                const uint32_t b0[2] = {b[0], b[1]}, b1[2] = {b[2], b[3]};
                mma_bf16(sc[nt], qf[kk], b0);
                mma_bf16(sc[nt], qf[kk + 1], b1);
            }
        }
    };

    // mask (causal, staged blocks only) and online softmax (log2 domain); P into A fragments
    auto softmax = [&](float (&sc)[8][4], int key0, uint32_t mask, uint32_t (&pf)[4][4]) {
        float bm[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int key = key0 + nt * 8 + 2 * tg + (c & 1);
                const bool staged = mask >> (nt >> 1) & 1u;
                const bool vis = staged && key < ((c >> 1) ? vis1 : vis0);
                sc[nt][c] = vis ? sc[nt][c] * p.scale_log2 : -INFINITY;
                bm[c >> 1] = fmaxf(bm[c >> 1], sc[nt][c]);
            }
        float alpha[2], mref[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            bm[r] = fmaxf(bm[r], __shfl_xor_sync(kFull, bm[r], 1));
            bm[r] = fmaxf(bm[r], __shfl_xor_sync(kFull, bm[r], 2));
            const float mn = fmaxf(m_run[r], bm[r]);
            mref[r] = mn == -INFINITY ? 0.f : mn;   // nothing visible to this row yet
            alpha[r] = fast_exp2(m_run[r] - mref[r]);
            m_run[r] = mn;
            l_run[r] *= alpha[r];
        }
#pragma unroll
        for (int nd = 0; nd < C::NDIM; ++nd) {
            oacc[nd][0] *= alpha[0];
            oacc[nd][1] *= alpha[0];
            oacc[nd][2] *= alpha[1];
            oacc[nd][3] *= alpha[1];
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {   // k-step = 16 keys (n-tiles 2kk, 2kk+1)
            const float p0 = fast_exp2(sc[nt][0] - mref[0]), p1 = fast_exp2(sc[nt][1] - mref[0]);
            const float p2 = fast_exp2(sc[nt][2] - mref[1]), p3 = fast_exp2(sc[nt][3] - mref[1]);
            l_run[0] += p0 + p1;
            l_run[1] += p2 + p3;
            pf[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16(p0, p1);
            pf[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16(p2, p3);
        }
    };

    // O += P V (V^T fragments by ldmatrix.trans; one block of 16 keys per k-step)
    auto pv = [&](uint32_t st, const uint32_t (&pf)[4][4]) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t vblk = st + kk * C::BLK;
#pragma unroll
            for (int nd = 0; nd < C::NDIM; nd += 2) {
                uint32_t b[4];
                ldsm_x4_trans(b, vblk + swz(kBS + (lane & 7) + ((lane >> 3) & 1) * 8, nd + (lane >> 4)));
                const uint32_t b0[2] = {b[0], b[1]}, b1[2] = {b[2], b[3]};
                mma_bf16(oacc[nd], pf[kk], b0);
                mma_bf16(oacc[nd + 1], pf[kk], b1);
            }
        }
    };

    // the last warp done with tile jj's stage refills it with tile jj + ring (no CTA-wide barrier)
    auto release = [&](int jj) {
        const int s = jj % kPrefillRing;
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            if (atomicAdd(&done_warps[s], 1) == kWarps - 1) {
                done_warps[s] = 0;
                if (jj + kPrefillRing < n_tiles) {
                    __threadfence_block();
                    fence_proxy_async_smem();
                    issue(jj + kPrefillRing);
                }
            }
        }
    };

    // one stage at a time (issuing the next stage's scores ahead of this stage's value
    // mixture measured slower on GB300: 73.6 vs 69.6 us for a 600-query chunk)
    bool timed_out = false;
    int j = 0;
    for (; j < n_tiles; ++j) {
        uint32_t st = 0, mask = 0;
        if (!acquire(j, st, mask)) {
            timed_out = true;
            break;
        }
        float sc[8][4];
        uint32_t pf[4][4];
        qk(st, sc);
        softmax(sc, j * kPrefillKeys, mask, pf);
        pv(st, pf);
        release(j);
    }

    if (timed_out) {   // record, then let copies already in flight land before the CTA exits
        if (lane == 0) {
            atomicOr(p.err, KVC_EBIT_TIMEOUT);
            for (int jj = j; jj < min(n_tiles, j + kPrefillRing); ++jj)
                (void)mbar_wait_bounded(smem_u32(&bars[jj % kPrefillRing]),
                                        static_cast<uint32_t>((jj / kPrefillRing) & 1), 100000000ull);
        }
        __syncthreads();
        return;
    }
    __syncthreads();   // no warp leaves while another may still refill a stage

    // ---- write out / lse of the real rows
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        float l = l_run[r];
        l += __shfl_xor_sync(kFull, l, 1);
        l += __shfl_xor_sync(kFull, l, 2);
        l_run[r] = l;
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int pos = pos0 + gq + 8 * r;
        if (pos >= n_q) continue;
        const float inv = 1.f / l_run[r];
        float *orow = p.out + (static_cast<size_t>(pos) * p.H_Q + hq) * D;
#pragma unroll
        for (int nd = 0; nd < C::NDIM; ++nd)
            *reinterpret_cast<float2 *>(orow + nd * 8 + 2 * tg) =
                make_float2(oacc[nd][2 * r] * inv, oacc[nd][2 * r + 1] * inv);
        if (p.lse && tg == 0) p.lse[static_cast<size_t>(pos) * p.H_Q + hq] = (m_run[r] + log2f(l_run[r])) * kLn2;
    }
}

// grid (1, KV head, position tile)
template <int D>
__global__ void __launch_bounds__(kThreads) prefill_kernel(const __grid_constant__ CUtensorMap tmap,
                                                           const DecodeParams p)
{
    prefill_cta<D>(tmap, p, blockIdx.z, blockIdx.y);
}

// In the mixed launch the query tiles keep 2 stages, and the kernel is held to 3
// CTAs per SM (the bf16 decode CTAs' occupancy).
constexpr int kMixedPrefillRing = 2;

// A decode step and a prefill chunk in one launch ("KV cache: Generation
// state, latency, and allocation" 21.3: chunked prefill beside decode):
// grid (split, KV head, decode units + prefill tiles).  The prefill tiles,
// compute-heavy and L2-resident, are spread evenly among the HBM-bound decode
// units (tile i of P sits at the z where floor(z * P / Z) steps), so the two
// kinds of work share the SMs.  FASTPRE: the prefill tiles run prefill_cta
// (bf16 pools, groups of at most 4 query heads); otherwise the split kernel's
// causal tiles.
template <int D, int NT, int KIND, bool PSPLIT, bool FASTPRE>
__global__ void __launch_bounds__(kThreads, FASTPRE ? 3 : 1) mixed_kernel(const __grid_constant__ CUtensorMap tmap,
                                                         const DecodeParams pd, const DecodeParams pp)
{
    allow_dependent_launch();
    const int z = blockIdx.z;
    const int64_t Z = gridDim.z, P = pp.B;
    const int before = static_cast<int>((static_cast<int64_t>(z) * P) / Z);
    const int upto = static_cast<int>((static_cast<int64_t>(z + 1) * P) / Z);
    if (upto > before) {
        if constexpr (FASTPRE) {
            if (blockIdx.x == 0) prefill_cta<D, kMixedPrefillRing>(tmap, pp, before, blockIdx.y);
        } else if (static_cast<int>(blockIdx.x) < pp.max_splits) {
            decode_cta<D, 4, KIND, false, true>(tmap, pp, blockIdx.x, blockIdx.y, before);
        }
    } else if (static_cast<int>(blockIdx.x) < pd.max_splits) {
        decode_cta<D, NT, KIND, PSPLIT, false>(tmap, pd, blockIdx.x, blockIdx.y, z - before);
    }
}

template <const void *(*FN)(), int SMEM>
DecodeKernel configured_kernel()
{
    DecodeKernel r;
    r.fn = FN();
    r.smem = SMEM;
    r.ctas_per_sm = 0;
    if (cudaFuncSetAttribute(r.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, r.smem) == cudaSuccess) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, r.fn, kThreads, r.smem) == cudaSuccess) r.ctas_per_sm = n;
    }
    return r;
}

template <int D, int NT, int KIND, bool PSPLIT, bool FASTPRE>
const void *mixed_fn() { return reinterpret_cast<const void *>(&mixed_kernel<D, NT, KIND, PSPLIT, FASTPRE>); }

template <int D>
const void *prefill_fn() { return reinterpret_cast<const void *>(&prefill_kernel<D>); }

constexpr int cmax(int a, int b) { return a > b ? a : b; }

template <int D, int NT, int KIND, bool PSPLIT, bool FASTPRE>
DecodeKernel mixed_instance()
{
    constexpr int smem = cmax(cmax(decode_smem_bytes<D, NT, KIND>(), decode_smem_bytes<D, 4, KIND>()),
                              FASTPRE ? PrefillCfg<D, kMixedPrefillRing>::SMEM : 0);
    static DecodeKernel k = configured_kernel<&mixed_fn<D, NT, KIND, PSPLIT, FASTPRE>, smem>();
    return k;
}

template <int D>
DecodeKernel prefill_instance()
{
    static DecodeKernel k = configured_kernel<&prefill_fn<D>, PrefillCfg<D>::SMEM>();
    return k;
}

// Mixed-launch kernel for a pool kind and decode group size (fn nullptr: unsupported shape).
DecodeKernel select_mixed_bf16(int D, int g, bool fast_prefill);
DecodeKernel select_mixed_fp8(int D, int g);
DecodeKernel select_mixed_int4(int D, int g);
// The query-tiled prefill kernel for bf16 pools (fn nullptr: unsupported shape).
DecodeKernel select_prefill_bf16(int D, int g);

}  // namespace kvc
