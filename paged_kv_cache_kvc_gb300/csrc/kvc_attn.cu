// Decode / prefill attention entry points, split sizing and the split merge.
#include <algorithm>
#include <cmath>
#include <cstdlib>

#include "kvc_decode_tc.cuh"
#include "kvc_prefill.cuh"
#include "kvc_prefill_tc.cuh"

namespace kvc {

// Log-sum-exp merge of a sequence's split partials ("flash-decoding"):
//   M = max_s m_s,  L = sum_s 2^(m_s - M) l_s,  out = sum_s 2^(m_s - M) o_s / L,
//   lse = (M + log2 L) ln 2.
// Sequences with a single split were finished by the attention kernel.
// grid (H_Q, query positions): one CTA per output row.  The merge is a few
// kilobytes per row, so its time is memory latency: every thread issues its
// loads of (m, l) and of up to kMergePre partial rows at once, before the
// sequence's length (and so its split count) is known -- every slot below
// max_splits lies inside the partials buffer, and slots past the split count are
// masked out by selection.  The CTA then reduces M and L over the splits, keeps
// the weights 2^(m_s - M) in shared memory (up to kMergeWeights splits; past that
// they are recomputed), and its D/4 float4 columns x (128 / (D/4)) split groups
// sum the partials before the groups are added.
// It is launched as a programmatic dependent of the attention kernel, so its
// CTAs are scheduled while that kernel drains; griddepcontrol.wait holds them
// until the attention kernel has finished and its partials are visible.
constexpr int kMergeWeights = 1024;
constexpr int kMergePre = 12;   // partial rows a thread loads up front

__device__ __forceinline__ float block_reduce_128(float v, bool is_max, float *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float t = __shfl_xor_sync(0xFFFFFFFFu, v, o);
        v = is_max ? fmaxf(v, t) : v + t;
    }
    __syncthreads();   // red is free
    if (lane == 0) red[warp] = v;
    __syncthreads();
    return is_max ? fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])) : (red[0] + red[1]) + (red[2] + red[3]);
}

__device__ __forceinline__ float4 fma4(float e, const float4 &o, float4 acc)
{
    acc.x = fmaf(e, o.x, acc.x);
    acc.y = fmaf(e, o.y, acc.y);
    acc.z = fmaf(e, o.z, acc.z);
    acc.w = fmaf(e, o.w, acc.w);
    return acc;
}

template <int D>
__global__ void __launch_bounds__(128) merge_kernel(const DecodeParams p)
{
    constexpr int ND4 = D / 4, G = 128 / ND4;
    static_assert(ND4 <= 128 && 128 % ND4 == 0, "D/4 float4 columns must divide the CTA");
    __shared__ float red[4];
    __shared__ float wsh[kMergeWeights];
    __shared__ float4 part[128];
    const int hq = blockIdx.x, pos = blockIdx.y, tid = threadIdx.x;
    const int d4 = tid % ND4, grp = tid / ND4;
    allow_dependent_launch();            // the next step's attention may be scheduled (it waits for this grid)
    int len = seq_len(p, pos / p.ppu);   // a caller input: read before the wait
    grid_dependency_wait();

    const int S = p.max_splits;
    const size_t bq = static_cast<size_t>(pos) * p.H_Q + hq;
    const float2 *ml = p.part_ml + bq * S;
    const float4 *po = reinterpret_cast<const float4 *>(p.part_o + bq * S * D) + d4;
    const float2 mv = tid < S ? ml[tid] : make_float2(0.f, 0.f);
    float4 o[kMergePre];
#pragma unroll
    for (int i = 0; i < kMergePre; ++i) {
        const int s = grp + G * i;
        o[i] = s < S ? po[static_cast<size_t>(s) * ND4] : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    if (len < 0 || static_cast<int64_t>(len) > static_cast<int64_t>(p.max_blocks) * kBS) len = 0;
    const int nblk = (len + kBS - 1) / kBS;
    const int ns = min((nblk + p.chunk - 1) / p.chunk, S);
    if (ns <= 1) return;   // uniform over the CTA

    float m = tid < ns ? mv.x : -INFINITY;
    for (int s = tid + 128; s < ns; s += 128) m = fmaxf(m, ml[s].x);
    const float M = block_reduce_128(m, true, red);
    const float Mref = M == -INFINITY ? 0.f : M;   // no visible position at all (device-detected errors)
    float l = 0.f;
    if (tid < ns) {
        const float e = fast_exp2(mv.x - Mref);
        l = e * mv.y;
        wsh[tid] = e;
    }
    for (int s = tid + 128; s < ns; s += 128) {
        const float2 v = ml[s];
        const float e = fast_exp2(v.x - Mref);
        l += e * v.y;
        if (s < kMergeWeights) wsh[s] = e;
    }
    const float L = block_reduce_128(l, false, red);   // its barriers also publish wsh

    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kMergePre; ++i) {
        const int s = grp + G * i;
        if (s < ns) acc = fma4(wsh[s], o[i], acc);
    }
    for (int s = grp + G * kMergePre; s < ns; s += G) {
        const float e = s < kMergeWeights ? wsh[s] : fast_exp2(ml[s].x - Mref);
        acc = fma4(e, po[static_cast<size_t>(s) * ND4], acc);
    }
    part[tid] = acc;
    __syncthreads();
    if (grp == 0) {
#pragma unroll
        for (int g2 = 1; g2 < G; ++g2) {
            const float4 v = part[g2 * ND4 + d4];
            acc.x += v.x;
            acc.y += v.y;
            acc.z += v.z;
            acc.w += v.w;
        }
        const float inv = 1.f / L;
        reinterpret_cast<float4 *>(p.out + bq * D)[d4] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
    if (tid == 0 && p.lse) p.lse[bq] = (M + log2f(L)) * kLn2;
}

// Blocks per split.  Sequences are independent and every CTA reads only its
// own blocks, so the kernel is bound by HBM once enough bytes are in flight;
// each CTA keeps 4 warps x (R - 1) stages in flight, so HBM wants more CTAs
// than one per resident slot.  Measured on GB300: about 1.7 CTAs per resident
// slot is best (a split costs a partial write and the merge).  No split is
// longer than kMaxChunk blocks, so that in a batch of unequal lengths the
// longest sequences do not set the launch's length (GB300, 64 sequences of
// log-uniform lengths 1 200..32 768: 299 us with 1 024-block splits, 253 us
// with 256-block splits); the hardware hands the many CTAs to SMs as they
// free, which also evens out SMs that stream at different rates.  Splits of
// one sequence are equal to within 4 blocks; a split holds at least 16 blocks
// (x the query n-tiles: a split's partials grow with the group size).
// KVC_SPLIT_CHUNK overrides (rounded up to 4).
constexpr int kMaxChunk = 288;

void choose_split(const kvc_pool *pool, int units, int max_blocks, int ctas_per_sm, int *chunk, int *max_splits,
                  int n_tiles)
{
    int ch = 0;
    if (const char *e = std::getenv("KVC_SPLIT_CHUNK")) ch = std::atoi(e);
    if (ch <= 0) {
        const double slots = static_cast<double>(pool->num_sms) * (ctas_per_sm > 0 ? ctas_per_sm : 1);
        long ns = units > 0 ? std::lround(1.7 * slots / units) : 1;
        ns = std::max(ns, static_cast<long>((max_blocks + kMaxChunk - 1) / kMaxChunk));
        if (ns < 1) ns = 1;
        ch = static_cast<int>((max_blocks + ns - 1) / ns);
        if (ch < 16 * n_tiles) ch = 16 * n_tiles;
    }
    ch = (ch + 3) & ~3;
    *chunk = ch;
    *max_splits = (max_blocks + ch - 1) / ch;
}

// The last split CTA of a unit merges its partials in the kernel while that is a
// small job (query columns x splits partial rows); larger merges run as merge_kernel.
static int merge_rows_limit()
{
    const char *e = std::getenv("KVC_MERGE_ROWS");
    return e ? std::min(std::atoi(e), kMergeRowsMax) : 64;
}

// The workspace holds the arrival counters at its front, at a fixed place
// whatever the batch (every launch leaves them at zero, so a later launch of
// another shape may use them), then the partials.  It grows by reallocation
// (zeroed); nothing in it outlives a launch except the zeroed counters.
static size_t counter_region(size_t n) { return (n * sizeof(uint32_t) + 255) & ~size_t(255); }

static kvc_status ensure_workspace(kvc_pool *pool, size_t counters, size_t bytes)
{
    if (counters <= pool->ws_counters && bytes <= pool->ws_bytes) return KVC_OK;
    counters = std::max(counters, pool->ws_counters);
    bytes = std::max(bytes, pool->ws_bytes);
    if (pool->ws) {
        cudaError_t e = cudaFree(pool->ws);
        pool->ws = nullptr;
        pool->ws_bytes = pool->ws_counters = 0;
        if (e != cudaSuccess) return cuda_status(e);
    }
    const size_t total = counter_region(counters) + bytes;
    if (cudaMalloc(&pool->ws, total) != cudaSuccess) {
        (void)cudaGetLastError();
        pool->ws = nullptr;
        return KVC_ERR_OOM;
    }
    pool->ws_bytes = bytes;
    pool->ws_counters = counters;
    return cuda_status(cudaMemset(pool->ws, 0, total));   // the arrival counters start at zero
}

static uint32_t *ws_counters(const kvc_pool *pool) { return static_cast<uint32_t *>(pool->ws); }
static float *ws_data(const kvc_pool *pool)
{
    return reinterpret_cast<float *>(static_cast<uint8_t *>(pool->ws) + counter_region(pool->ws_counters));
}

// split partials: o [units'][H_Q][splits][D], then (max, sum) [units'][H_Q][splits]
static size_t workspace_bytes(int B, int H_Q, int max_splits, int D)
{
    const size_t n = static_cast<size_t>(B) * H_Q * max_splits;
    return n * D * sizeof(float) + n * sizeof(float2);
}

// Launches a decode attention kernel as a programmatic dependent of whatever precedes it
// on the stream.  The kernels wait (griddepcontrol.wait) for that grid before their first
// global access, so their launch and set-up overlap its tail: in a decode loop, the
// previous step's attention or merge.  When what precedes it is not a kernel, the launch
// behaves as an ordinary one.
static cudaError_t launch_programmatic_dependent(const void *fn, dim3 grid, dim3 block, int smem, cudaStream_t stream,
                                                 void **args)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

kvc_status run_decode(const kvc_pool *cpool, DecodeParams &p, const DecodeKernel &k, cudaStream_t stream)
{
    kvc_pool *pool = const_cast<kvc_pool *>(cpool);
    if (!k.fn || k.ctas_per_sm <= 0) return KVC_ERR_CUDA;
    choose_split(pool, p.B * p.H_KV, p.max_blocks, k.ctas_per_sm, &p.chunk, &p.max_splits, n_tiles(p.ppu * p.g));
    if (p.max_splits > 65535) return KVC_ERR_UNSUPPORTED;
    if (p.max_splits > 1) {
        kvc_status st = ensure_workspace(pool, static_cast<size_t>(p.B) * p.H_KV,
                                         workspace_bytes(p.n_pos, p.H_Q, p.max_splits, pool->D));
        if (st != KVC_OK) return st;
        const size_t n = static_cast<size_t>(p.n_pos) * p.H_Q * p.max_splits;
        p.part_o = ws_data(pool);
        p.part_ml = reinterpret_cast<float2 *>(p.part_o + n * pool->D);
        // the last split CTA merges its group in the kernel when that is a small job (g * splits
        // partial rows); otherwise one merge CTA per (sequence, query head) does it afterwards
        p.counters = (p.ppu * p.g * p.max_splits <= merge_rows_limit()) ? ws_counters(pool) : nullptr;
    } else {
        p.part_o = nullptr;
        p.part_ml = nullptr;
        p.counters = nullptr;
    }
    void *args[] = {const_cast<CUtensorMap *>(&pool->tmap), &p};
    const cudaError_t e =
        launch_programmatic_dependent(k.fn, dim3(p.max_splits, p.H_KV, p.B), dim3(kThreads), k.smem, stream, args);
    if (e != cudaSuccess) return cuda_status(e);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (p.max_splits > 1 && !p.counters) return launch_split_merge(p, pool->D, stream);
    return KVC_OK;
}

// The query-tiled prefill kernel serves bf16 pools with groups of at most 4 query
// heads (KVC_PREFILL_PPU, which sizes the split kernel's causal tiles, selects those).
static bool fast_prefill(const kvc_pool *pool, int g)
{
    return pool->dtype == KVC_BF16 && g <= 4 && (pool->D == 64 || pool->D == 128) && !std::getenv("KVC_PREFILL_PPU");
}

static kvc_status launch_prefill_fast(kvc_pool *pool, DecodeParams &p, cudaStream_t stream)
{
    const DecodeKernel k = select_prefill_bf16(pool->D, p.g);
    if (!k.fn || k.ctas_per_sm <= 0) return KVC_ERR_UNSUPPORTED;
    if (p.B > 65535) return KVC_ERR_UNSUPPORTED;
    p.chunk = p.max_blocks;
    p.max_splits = 1;
    void *args[] = {const_cast<CUtensorMap *>(&pool->tmap), &p};
    const cudaError_t e = cudaLaunchKernel(k.fn, dim3(1, pool->H_KV, p.B), dim3(kThreads), args, k.smem, stream);
    if (e != cudaSuccess) return cuda_status(e);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return KVC_OK;
}

// A decode step (pd) and a prefill chunk (pp) in one mixed_kernel launch; each
// part keeps the split plan it would get alone and its own partials and counters.
static kvc_status run_mixed(kvc_pool *pool, DecodeParams &pd, DecodeParams &pp, const DecodeKernel &k,
                            bool fast_prefill, cudaStream_t stream)
{
    if (!k.fn || k.ctas_per_sm <= 0) return KVC_ERR_UNSUPPORTED;
    choose_split(pool, pd.B * pd.H_KV, pd.max_blocks, k.ctas_per_sm, &pd.chunk, &pd.max_splits, n_tiles(pd.g));
    if (fast_prefill) {   // query tiles read their whole causal range: no splits
        pp.chunk = pp.max_blocks;
        pp.max_splits = 1;
    } else {
        choose_split(pool, pp.B * pp.H_KV, pp.max_blocks, k.ctas_per_sm, &pp.chunk, &pp.max_splits,
                     n_tiles(pp.ppu * pp.g));
    }
    const int splits = std::max(pd.max_splits, pp.max_splits);
    if (splits > 65535 || static_cast<int64_t>(pd.B) + pp.B > 65535) return KVC_ERR_UNSUPPORTED;
    const size_t ud = static_cast<size_t>(pd.B) * pd.H_KV, up = static_cast<size_t>(pp.B) * pp.H_KV;
    const size_t nd = pd.max_splits > 1 ? static_cast<size_t>(pd.n_pos) * pd.H_Q * pd.max_splits : 0;
    const size_t np = pp.max_splits > 1 ? static_cast<size_t>(pp.n_pos) * pp.H_Q * pp.max_splits : 0;
    const size_t row = static_cast<size_t>(pool->D) * sizeof(float) + sizeof(float2);
    kvc_status st = ensure_workspace(pool, ud + up, (nd + np) * row + 256);
    if (st != KVC_OK) return st;
    float *data = ws_data(pool);
    pd.part_o = nd ? data : nullptr;
    pd.part_ml = nd ? reinterpret_cast<float2 *>(data + nd * pool->D) : nullptr;
    pd.counters = (nd && pd.ppu * pd.g * pd.max_splits <= merge_rows_limit()) ? ws_counters(pool) : nullptr;
    float *data_p = data + ((nd * pool->D + nd * 2 + 63) & ~static_cast<size_t>(63));   // 256-byte aligned
    pp.part_o = np ? data_p : nullptr;
    pp.part_ml = np ? reinterpret_cast<float2 *>(data_p + np * pool->D) : nullptr;
    pp.counters = (np && pp.ppu * pp.g * pp.max_splits <= merge_rows_limit()) ? ws_counters(pool) + ud : nullptr;
    void *args[] = {const_cast<CUtensorMap *>(&pool->tmap), &pd, &pp};
    cudaError_t e = cudaLaunchKernel(k.fn, dim3(splits, pool->H_KV, pd.B + pp.B), dim3(kThreads), args, k.smem,
                                     stream);
    if (e != cudaSuccess) return cuda_status(e);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (nd && !pd.counters && (st = launch_split_merge(pd, pool->D, stream)) != KVC_OK) return st;
    if (np && !pp.counters && (st = launch_split_merge(pp, pool->D, stream)) != KVC_OK) return st;
    return KVC_OK;
}

// Splits of the tensor-memory decode kernels: about one CTA per resident slot (one
// per SM; the ring keeps ~100 KiB in flight, so more CTAs than slots only add split
// partials), the longest row's blocks shared evenly among them, rounded up to a
// multiple of `unit` blocks.  A split walks 128-token tiles from its first block, so
// the kernels take any split; the e4m3 kernel runs fastest with even shares (unit 1:
// the CTA with the most bytes stays close to the mean), the bf16 kernel with whole
// tiles (unit 8; even shares measured 8 % slower).  KVC_SPLIT_CHUNK overrides
// (blocks per split, rounded up to the unit).
void choose_split_tc(const kvc_pool *pool, int units, int max_blocks, int ctas_per_sm, int unit, int *chunk,
                     int *max_splits)
{
    const int tiles = (max_blocks + kTcBlocks - 1) / kTcBlocks;
    unit = std::max(unit, 1);
    int cb = 0;
    if (const char *e = std::getenv("KVC_SPLIT_CHUNK")) cb = std::atoi(e);
    if (cb <= 0) {
        const double slots = static_cast<double>(pool->num_sms) * (ctas_per_sm > 0 ? ctas_per_sm : 1);
        long ns = units > 0 ? std::lround(slots / units) : 1;
        ns = std::max(1L, std::min(ns, static_cast<long>(tiles)));
        cb = static_cast<int>((max_blocks + ns - 1) / ns);
    }
    *chunk = (cb + unit - 1) / unit * unit;
    *max_splits = (max_blocks + *chunk - 1) / *chunk;
}

// The tensor-memory kernels serve decode steps of 32-head groups on d_h 128 bf16 and
// e4m3 pools (KVC_TC=0 selects the split kernel for them).
DecodeKernel tc_kernel_for(const kvc_pool *pool, const DecodeParams &p)
{
    const char *e = std::getenv("KVC_TC");
    if ((e && e[0] == '0') || !p.lens || p.ppu != 1 || pool->bs != kBS) return DecodeKernel{nullptr, 0, 0};
    const DecodeKernel k = select_decode_tc(pool->D, p.g, pool->dtype);
    if (!k.fn || !(k.tmap16 ? pool->tmap16_ok : pool->tmap_ok)) return DecodeKernel{nullptr, 0, 0};
    return k;
}

static kvc_status run_decode_tc(kvc_pool *pool, DecodeParams &p, const DecodeKernel &k, cudaStream_t stream)
{
    if (k.ctas_per_sm <= 0) return KVC_ERR_CUDA;
    choose_split_tc(pool, p.B * p.H_KV, p.max_blocks, k.ctas_per_sm, k.split_unit, &p.chunk, &p.max_splits);
    if (p.max_splits > 65535) return KVC_ERR_UNSUPPORTED;
    p.counters = nullptr;   // splits are merged by merge_kernel
    p.part_o = nullptr;
    p.part_ml = nullptr;
    if (p.max_splits > 1) {
        kvc_status st = ensure_workspace(pool, static_cast<size_t>(p.B) * p.H_KV,
                                         workspace_bytes(p.n_pos, p.H_Q, p.max_splits, pool->D));
        if (st != KVC_OK) return st;
        const size_t n = static_cast<size_t>(p.n_pos) * p.H_Q * p.max_splits;
        p.part_o = ws_data(pool);
        p.part_ml = reinterpret_cast<float2 *>(p.part_o + n * pool->D);
    }
    void *args[] = {const_cast<CUtensorMap *>(k.tmap16 ? &pool->tmap16 : &pool->tmap), &p};
    const cudaError_t e =
        launch_programmatic_dependent(k.fn, dim3(p.max_splits, p.H_KV, p.B), dim3(k.threads), k.smem, stream, args);
    if (e != cudaSuccess) return cuda_status(e);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (p.max_splits > 1) return launch_split_merge(p, pool->D, stream);
    return KVC_OK;
}

// The tensor-memory prefill kernel serves bf16 pools of d_h 64 or 128, every group
// size (KVC_TC=0, or KVC_PREFILL_PPU for the split kernel's causal tiles, select
// the other kernels).
static DecodeKernel prefill_tc_for(const kvc_pool *pool)
{
    const char *e = std::getenv("KVC_TC");
    if ((e && e[0] == '0') || std::getenv("KVC_PREFILL_PPU") || !pool->tmap16_ok || pool->bs != kBS)
        return DecodeKernel{nullptr, 0, 0};
    return select_prefill_tc(pool->D, pool->dtype);
}

// grid (1, KV head, tile of 128 / g positions).  dependent: launched as a
// programmatic dependent of the kernel before it on the stream, whose CTAs it may
// run beside (it reads nothing that kernel writes and never waits on it).
static kvc_status launch_prefill_tc(const kvc_pool *pool, DecodeParams &p, const DecodeKernel &k, bool dependent,
                                    cudaStream_t stream)
{
    if (k.ctas_per_sm <= 0) return KVC_ERR_CUDA;
    p.ppu = 128 / p.g;
    p.B = (p.n_pos + p.ppu - 1) / p.ppu;
    p.chunk = p.max_blocks;
    p.max_splits = 1;
    if (p.B > 65535) return KVC_ERR_UNSUPPORTED;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, pool->H_KV, p.B);
    cfg.blockDim = dim3(kPtThreads);
    cfg.dynamicSmemBytes = k.smem;
    cfg.stream = stream;
    cfg.attrs = dependent ? attr : nullptr;
    cfg.numAttrs = dependent ? 1 : 0;
    void *args[] = {const_cast<CUtensorMap *>(&pool->tmap16), &p};
    const cudaError_t e = cudaLaunchKernelExC(&cfg, k.fn, args);
    if (e != cudaSuccess) return cuda_status(e);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return KVC_OK;
}

static bool aligned(const void *ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

static kvc_status common_attn_checks(kvc_pool *pool, int32_t layer, const void *q, int32_t H_Q, const int32_t *bt,
                                     int32_t max_blocks, float *out, float *lse, float scale)
{
    if (!pool || !q || !bt || !out) return KVC_ERR_ARG;
    if (layer < 0 || layer >= pool->L) return KVC_ERR_ARG;
    if (H_Q <= 0 || H_Q % pool->H_KV != 0) return KVC_ERR_ARG;
    if (H_Q / pool->H_KV > 32) return KVC_ERR_UNSUPPORTED;
    if (pool->bs != kBS || !pool->tmap_ok) return KVC_ERR_UNSUPPORTED;
    if (max_blocks <= 0 || max_blocks > (1 << 26)) return KVC_ERR_ARG;
    if (!std::isfinite(scale)) return KVC_ERR_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || (lse && !aligned(lse, 4)) || !aligned(bt, 4)) return KVC_ERR_ARG;
    return check_device(pool);
}

static void fill_common(DecodeParams &p, const kvc_pool *pool, int32_t layer, const void *q, int32_t H_Q,
                        const int32_t *bt, int32_t max_blocks, float *out, float *lse, float scale)
{
    p.q = static_cast<const uint16_t *>(q);
    p.bt = bt;
    p.max_blocks = max_blocks;
    p.H_Q = H_Q;
    p.H_KV = pool->H_KV;
    p.g = H_Q / pool->H_KV;
    p.layer = layer;
    p.N = pool->N;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.s_k = pool->scales ? pool->scales + static_cast<size_t>(layer) * 2 * pool->H_KV * pool->D : nullptr;
    p.s_v = p.s_k ? p.s_k + static_cast<size_t>(pool->H_KV) * pool->D : nullptr;
    p.out = out;
    p.lse = lse;
    p.err = pool->err;
    p.pool = pool->base;   // the fused append's stores and the kernels' speculative L2 prefetch
    p.stall_loads = std::getenv("KVC_TEST_STALL") ? 1 : 0;
}

static kvc_status dispatch(kvc_pool *pool, DecodeParams &p, cudaStream_t stream)
{
    const DecodeKernel tc = tc_kernel_for(pool, p);
    if (tc.fn) return run_decode_tc(pool, p, tc, stream);
    if (pool->dtype == KVC_FP8_E4M3) return launch_decode_fp8(pool, p, stream);
    if (pool->dtype == KVC_INT4) return launch_decode_int4(pool, p, stream);
    return launch_decode_bf16(pool, p, stream);
}

}  // namespace kvc

using namespace kvc;

extern "C" kvc_status kvc_decode_attn(kvc_pool *pool, int32_t layer, const void *q, int32_t num_q_heads,
                                      const int32_t *block_tables, int32_t max_blocks, const int32_t *seq_lens,
                                      int32_t B, float *out, float *lse, float scale, kvc_stream_t stream)
{
    if (B < 0 || B > 65535) return KVC_ERR_ARG;
    if (B == 0) return pool ? KVC_OK : KVC_ERR_ARG;
    if (!seq_lens || !aligned(seq_lens, 4)) return KVC_ERR_ARG;
    kvc_status st = common_attn_checks(pool, layer, q, num_q_heads, block_tables, max_blocks, out, lse, scale);
    if (st != KVC_OK) return st;
    DecodeParams p{};
    fill_common(p, pool, layer, q, num_q_heads, block_tables, max_blocks, out, lse, scale);
    p.lens = seq_lens;
    p.bt_stride = max_blocks;
    p.len_base = 0;
    p.B = B;
    p.ppu = 1;
    p.n_pos = B;
    return dispatch(pool, p, static_cast<cudaStream_t>(stream));
}

extern "C" kvc_status kvc_decode_step(kvc_pool *pool, int32_t layer, const void *q, int32_t num_q_heads,
                                      const int32_t *block_tables, int32_t max_blocks, const int32_t *seq_lens,
                                      int32_t B, const void *k_new, const void *v_new, float *out, float *lse,
                                      float scale, kvc_stream_t stream)
{
    if (B < 0 || B > 65535) return KVC_ERR_ARG;
    if (B == 0) return pool ? KVC_OK : KVC_ERR_ARG;
    if (!seq_lens || !aligned(seq_lens, 4) || !k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16))
        return KVC_ERR_ARG;
    kvc_status st = common_attn_checks(pool, layer, q, num_q_heads, block_tables, max_blocks, out, lse, scale);
    if (st != KVC_OK) return st;
    DecodeParams p{};
    fill_common(p, pool, layer, q, num_q_heads, block_tables, max_blocks, out, lse, scale);
    p.lens = seq_lens;
    p.bt_stride = max_blocks;
    p.len_base = 0;
    p.B = B;
    p.ppu = 1;
    p.n_pos = B;
    p.k_new = static_cast<const uint16_t *>(k_new);
    p.v_new = static_cast<const uint16_t *>(v_new);
    p.pool = pool->base;
    return dispatch(pool, p, static_cast<cudaStream_t>(stream));
}

extern "C" kvc_status kvc_prefill_attn(kvc_pool *pool, int32_t layer, const void *q, int32_t n_q,
                                       int32_t num_q_heads, const int32_t *block_table_row, int32_t max_blocks,
                                       int32_t q_start, float *out, float *lse, float scale, kvc_stream_t stream)
{
    if (n_q < 0 || n_q > 65535 || q_start < 0) return KVC_ERR_ARG;
    if (n_q == 0) return pool ? KVC_OK : KVC_ERR_ARG;
    kvc_status st = common_attn_checks(pool, layer, q, num_q_heads, block_table_row, max_blocks, out, lse, scale);
    if (st != KVC_OK) return st;
    if (static_cast<int64_t>(q_start) + n_q > static_cast<int64_t>(max_blocks) * kBS) return KVC_ERR_RANGE;
    DecodeParams p{};
    fill_common(p, pool, layer, q, num_q_heads, block_table_row, max_blocks, out, lse, scale);
    // query i reads q_start + i + 1 positions of the same row; a unit (CTA
    // column group) takes ppu consecutive queries x the g heads of a KV head,
    // so each staged block serves ppu queries.  KVC_PREFILL_PPU overrides.
    p.lens = nullptr;
    p.bt_stride = 0;
    p.len_base = q_start;
    // the chunk reads positions < q_start + n_q: plan splits over those blocks only
    p.max_blocks = static_cast<int32_t>((static_cast<int64_t>(q_start) + n_q + kBS - 1) / kBS);
    p.n_pos = n_q;
    const DecodeKernel tc = prefill_tc_for(pool);
    if (tc.fn) return launch_prefill_tc(pool, p, tc, false, static_cast<cudaStream_t>(stream));
    if (fast_prefill(pool, p.g)) {   // query tiles of 64 / g positions x g heads on the M dimension
        p.ppu = 64 / p.g;
        p.B = (n_q + p.ppu - 1) / p.ppu;
        return launch_prefill_fast(pool, p, static_cast<cudaStream_t>(stream));
    }
    int ppu = 32 / p.g;     // measured on GB300 (600-query chunk, g = 4): 1 -> 346 us, 4 -> 143 us, 8 -> 135 us
    if (const char *e = std::getenv("KVC_PREFILL_PPU")) ppu = std::atoi(e);
    ppu = std::max(1, std::min(ppu, 32 / p.g));
    p.ppu = ppu;
    p.B = (n_q + ppu - 1) / ppu;
    return dispatch(pool, p, static_cast<cudaStream_t>(stream));
}

extern "C" kvc_status kvc_mixed_step(kvc_pool *pool, int32_t layer, const void *q, int32_t num_q_heads,
                                     const int32_t *block_tables, int32_t max_blocks, const int32_t *seq_lens,
                                     int32_t B, const void *k_new, const void *v_new, float *out, float *lse,
                                     const void *prefill_q, int32_t n_q, const int32_t *prefill_block_table_row,
                                     int32_t prefill_max_blocks, int32_t q_start, float *prefill_out,
                                     float *prefill_lse, float scale, kvc_stream_t stream)
{
    if (B < 0 || B > 65535 || n_q < 0 || n_q > 65535 || q_start < 0) return KVC_ERR_ARG;
    if (n_q == 0)
        return kvc_decode_step(pool, layer, q, num_q_heads, block_tables, max_blocks, seq_lens, B, k_new, v_new, out,
                               lse, scale, stream);
    if (B == 0)
        return kvc_prefill_attn(pool, layer, prefill_q, n_q, num_q_heads, prefill_block_table_row,
                                prefill_max_blocks, q_start, prefill_out, prefill_lse, scale, stream);
    if (!seq_lens || !aligned(seq_lens, 4) || !k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16))
        return KVC_ERR_ARG;
    kvc_status st = common_attn_checks(pool, layer, q, num_q_heads, block_tables, max_blocks, out, lse, scale);
    if (st != KVC_OK) return st;
    st = common_attn_checks(pool, layer, prefill_q, num_q_heads, prefill_block_table_row, prefill_max_blocks,
                            prefill_out, prefill_lse, scale);
    if (st != KVC_OK) return st;
    if (static_cast<int64_t>(q_start) + n_q > static_cast<int64_t>(prefill_max_blocks) * kBS) return KVC_ERR_RANGE;
    if (const DecodeKernel tc = prefill_tc_for(pool); tc.fn) {
        // the decode step, then the chunk on the tensor-memory prefill kernel as a programmatic
        // dependent: its CTAs take SMs as the decode CTAs drain, and it never waits on them
        st = kvc_decode_step(pool, layer, q, num_q_heads, block_tables, max_blocks, seq_lens, B, k_new, v_new, out, lse,
                             scale, stream);
        if (st != KVC_OK) return st;
        DecodeParams pt{};
        fill_common(pt, pool, layer, prefill_q, num_q_heads, prefill_block_table_row, prefill_max_blocks, prefill_out,
                    prefill_lse, scale);
        pt.lens = nullptr;
        pt.bt_stride = 0;
        pt.len_base = q_start;
        pt.max_blocks = static_cast<int32_t>((static_cast<int64_t>(q_start) + n_q + kBS - 1) / kBS);
        pt.n_pos = n_q;
        return launch_prefill_tc(pool, pt, tc, true, static_cast<cudaStream_t>(stream));
    }
    DecodeParams pd{};
    fill_common(pd, pool, layer, q, num_q_heads, block_tables, max_blocks, out, lse, scale);
    pd.lens = seq_lens;
    pd.bt_stride = max_blocks;
    pd.B = B;
    pd.ppu = 1;
    pd.n_pos = B;
    pd.k_new = static_cast<const uint16_t *>(k_new);
    pd.v_new = static_cast<const uint16_t *>(v_new);
    pd.pool = pool->base;
    DecodeParams pp{};
    fill_common(pp, pool, layer, prefill_q, num_q_heads, prefill_block_table_row, prefill_max_blocks, prefill_out,
                prefill_lse, scale);
    pp.lens = nullptr;
    pp.bt_stride = 0;
    pp.len_base = q_start;
    pp.max_blocks = static_cast<int32_t>((static_cast<int64_t>(q_start) + n_q + kBS - 1) / kBS);
    const bool fast = fast_prefill(pool, pp.g);
    pp.ppu = fast ? 64 / pp.g : std::max(1, 32 / pp.g);
    pp.n_pos = n_q;
    pp.B = (n_q + pp.ppu - 1) / pp.ppu;
    DecodeKernel k{nullptr, 0, 0};
    if (pool->dtype == KVC_FP8_E4M3) k = select_mixed_fp8(pool->D, pd.g);
    else if (pool->dtype == KVC_INT4) k = select_mixed_int4(pool->D, pd.g);
    else k = select_mixed_bf16(pool->D, pd.g, fast);
    if (!k.fn) {   // no mixed instance for this shape: the two launches in order
        st = kvc_decode_step(pool, layer, q, num_q_heads, block_tables, max_blocks, seq_lens, B, k_new, v_new, out,
                             lse, scale, stream);
        if (st != KVC_OK) return st;
        return kvc_prefill_attn(pool, layer, prefill_q, n_q, num_q_heads, prefill_block_table_row,
                                prefill_max_blocks, q_start, prefill_out, prefill_lse, scale, stream);
    }
    return run_mixed(pool, pd, pp, k, fast, static_cast<cudaStream_t>(stream));
}

extern "C" kvc_status kvc_pool_reserve(kvc_pool *pool, int32_t max_batch, int32_t num_q_heads, int32_t max_blocks)
{
    if (!pool || max_batch < 0 || num_q_heads <= 0 || max_blocks <= 0) return KVC_ERR_ARG;
    kvc_status st = check_device(pool);
    if (st != KVC_OK) return st;
    // the largest split count any batch of this size can get is the 16-block floor
    const int max_splits = (max_blocks + 15) / 16;
    const size_t units = static_cast<size_t>(max_batch) * pool->H_KV;
    return ensure_workspace(pool, units, workspace_bytes(max_batch, num_q_heads, max_splits, pool->D));
}

namespace kvc {

// Launch the split merge on its own (partials already written by the decode kernel).
// merge_kernel as a programmatic dependent of the kernel before it on the stream
kvc_status launch_split_merge(const DecodeParams &p, int D, cudaStream_t stream)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.H_Q, p.n_pos);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (D == 64) e = cudaLaunchKernelEx(&cfg, merge_kernel<64>, p);
    else if (D == 128) e = cudaLaunchKernelEx(&cfg, merge_kernel<128>, p);
    else return KVC_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return cuda_status(e);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return KVC_OK;
}

}  // namespace kvc
