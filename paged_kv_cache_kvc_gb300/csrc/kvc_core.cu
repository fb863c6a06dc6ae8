// Pool management, the append / token-write scatter kernel, fp8 calibration
// and the host utilities of libkvc.
#include <cmath>
#include <cstring>
#include <cudaTypedefs.h>
#include <new>

#include "kvc_internal.h"
#include "kvc_ptx.cuh"

namespace kvc {

std::atomic<uint64_t> g_launches{0};

kvc_status cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return KVC_OK;
    if (e == cudaErrorMemoryAllocation) return KVC_ERR_OOM;
    return KVC_ERR_CUDA;
}

kvc_status check_device(const kvc_pool *pool)
{
    int d = -1;
    if (cudaGetDevice(&d) != cudaSuccess) return KVC_ERR_CUDA;
    return d == pool->device ? KVC_OK : KVC_ERR_ARG;
}

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// ------------------------------------------------------------------ scatter
// "KV cache: Generation state, latency, and allocation" Eq. 21.6 and
// Table 21.1 steps 1-2: token t of sequence b goes to block table[b][t / bs],
// slot t mod bs, keys and values of every KV head.  One thread moves one
// 16-byte chunk (8 channels) of one row.
struct ScatterParams {
    uint8_t *base;
    int64_t N;
    int32_t bs, H_KV, D, s, layer;
    const int32_t *bt;
    int32_t max_blocks;
    const int32_t *start;   // [B] first position written
    const int32_t *cu;      // [B+1] token offsets, or nullptr: one token per sequence at row b
    const uint16_t *k, *v;  // bf16 [rows][H_KV][D]
    const float *scales;    // this layer's [2][H_KV][D] for e4m3 / int4, else nullptr
    int32_t bits;           // stored bits per element: 16, 8, 4
    uint32_t *err;
    int32_t tok_per_cta;
};

__global__ void __launch_bounds__(256) scatter_kernel(const ScatterParams p)
{
    const int b = blockIdx.y;
    int i0 = b, n = 1;
    if (p.cu) {
        i0 = __ldg(p.cu + b);
        n = __ldg(p.cu + b + 1) - i0;
    }
    const int t_lo = blockIdx.x * p.tok_per_cta;
    const int t_hi = min(n, t_lo + p.tok_per_cta);
    if (t_lo >= t_hi) return;
    const int start = __ldg(p.start + b);
    const int cpr = p.D / 8;                 // 16-byte chunks per row
    const int per_tok = 2 * p.H_KV * cpr;
    for (int idx = threadIdx.x; idx < (t_hi - t_lo) * per_tok; idx += blockDim.x) {
        const int ti = t_lo + idx / per_tok;
        int rem = idx % per_tok;
        const int kv = rem / (p.H_KV * cpr);
        rem -= kv * p.H_KV * cpr;
        const int h = rem / cpr, ch = rem - h * cpr;
        const int64_t t = static_cast<int64_t>(start) + ti;
        const bool first = (kv == 0 && h == 0 && ch == 0);
        if (start < 0 || t / p.bs >= p.max_blocks) {
            if (first) atomicOr(p.err, KVC_EBIT_RANGE);
            continue;
        }
        const int32_t phys = __ldg(p.bt + static_cast<int64_t>(b) * p.max_blocks + t / p.bs);
        if (phys < 0 || static_cast<int64_t>(phys) >= p.N) {
            if (first) atomicOr(p.err, KVC_EBIT_BAD_BLOCK);
            continue;
        }
        const int slot = static_cast<int>(t % p.bs);
        const uint16_t *src = (kv ? p.v : p.k) + (static_cast<int64_t>(i0 + ti) * p.H_KV + h) * p.D + ch * 8;
        const uint4 x = *reinterpret_cast<const uint4 *>(src);
        const int64_t e =
            ((((static_cast<int64_t>(p.layer) * p.N + phys) * p.H_KV + h) * 2 + kv) * p.bs + slot) * p.D + ch * 8;
        if (p.bits == 16) {
            *reinterpret_cast<uint4 *>(p.base + e * 2) = x;
        } else if (p.bits == 4) {   // rint(x / s) clamped to [-7, 7], nibble q + 8; channel 2j in the low nibble
            const float *sc = p.scales + (static_cast<int64_t>(kv) * p.H_KV + h) * p.D + ch * 8;
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
            uint32_t packed = 0u;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float f = (i & 1) ? bf16_hi(w[i >> 1]) : bf16_lo(w[i >> 1]);
                const float y = __fdiv_rn(f, __ldg(sc + i));
                const uint32_t q = isnan(y) ? 8u
                                            : static_cast<uint32_t>(static_cast<int>(fminf(fmaxf(rintf(y), -7.f), 7.f)) + 8);
                packed |= q << (4 * i);
            }
            *reinterpret_cast<uint32_t *>(p.base + e / 2) = packed;
        } else {
            const float *sc = p.scales + (static_cast<int64_t>(kv) * p.H_KV + h) * p.D + ch * 8;
            const uint32_t w[4] = {x.x, x.y, x.z, x.w};
            uint32_t packed[2] = {0u, 0u};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float f = (i & 1) ? bf16_hi(w[i >> 1]) : bf16_lo(w[i >> 1]);
                const uint32_t q = __nv_cvt_float_to_fp8(__fdiv_rn(f, __ldg(sc + i)), __NV_SATFINITE, __NV_E4M3);
                packed[i >> 2] |= q << (8 * (i & 3));
            }
            *reinterpret_cast<uint2 *>(p.base + e) = make_uint2(packed[0], packed[1]);
        }
    }
}

static bool aligned(const void *ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

static kvc_status scatter(kvc_pool *pool, int32_t layer, const int32_t *bt, int32_t max_blocks, const int32_t *start,
                          const int32_t *cu, int32_t B, int32_t max_tokens, const void *k, const void *v,
                          cudaStream_t stream)
{
    if (!pool) return KVC_ERR_ARG;
    if (B < 0 || B > 65535 || max_tokens < 0) return KVC_ERR_ARG;
    if (B == 0 || max_tokens == 0) return KVC_OK;
    if (layer < 0 || layer >= pool->L || max_blocks <= 0) return KVC_ERR_ARG;
    if (!bt || !start || !k || !v || !aligned(k, 16) || !aligned(v, 16) || !aligned(bt, 4) || !aligned(start, 4))
        return KVC_ERR_ARG;
    kvc_status st = check_device(pool);
    if (st != KVC_OK) return st;
    ScatterParams p{};
    p.base = pool->base;
    p.N = pool->N;
    p.bs = pool->bs;
    p.H_KV = pool->H_KV;
    p.D = pool->D;
    p.s = pool->s;
    p.layer = layer;
    p.bt = bt;
    p.max_blocks = max_blocks;
    p.start = start;
    p.cu = cu;
    p.k = static_cast<const uint16_t *>(k);
    p.v = static_cast<const uint16_t *>(v);
    p.scales = pool->scales ? pool->scales + static_cast<size_t>(layer) * 2 * pool->H_KV * pool->D : nullptr;
    p.err = pool->err;
    p.bits = pool->bits;
    const int per_tok = 2 * pool->H_KV * (pool->D / 8);
    p.tok_per_cta = per_tok >= 4096 ? 1 : 4096 / per_tok;
    const int gx = (max_tokens + p.tok_per_cta - 1) / p.tok_per_cta;
    scatter_kernel<<<dim3(gx, B), 256, 0, stream>>>(p);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_status(e);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return KVC_OK;
}

// ------------------------------------------------------------------ fp8 calibration
__global__ void absmax_kernel(const uint16_t *x, int64_t n_tokens, int HD, int tok_per_cta, float *amax)
{
    const int64_t t0 = static_cast<int64_t>(blockIdx.x) * tok_per_cta;
    const int64_t t1 = min(n_tokens, t0 + tok_per_cta);
    for (int c = blockIdx.y * blockDim.x + threadIdx.x; c < HD; c += blockDim.x * gridDim.y) {
        float m = 0.f;
        for (int64_t t = t0; t < t1; ++t) m = fmaxf(m, fabsf(__uint_as_float(static_cast<uint32_t>(x[t * HD + c]) << 16)));
        atomicMax(reinterpret_cast<unsigned int *>(amax + c), __float_as_uint(m));   // m >= 0: orders as uint
    }
}

// scale = absmax / qmax (448: largest finite e4m3; 7: int4 range), 1 for an all-zero channel
__global__ void scales_from_absmax_kernel(const float *amax, float *scales, int n, float qmax)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) scales[i] = amax[i] > 0.f ? __fdiv_rn(amax[i], qmax) : 1.f;
}

__global__ void fill_kernel(float *x, float v, int n)
{
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) x[i] = v;
}

}  // namespace kvc

using namespace kvc;

// ------------------------------------------------------------------ C ABI
extern "C" uint64_t kvc_bytes(int64_t L, int64_t B, int64_t H_KV, int64_t T, int64_t d_h, int64_t s)
{
    // "KV cache: Generation state, latency, and allocation" Eq. 21.2
    const int64_t f[7] = {2, L, B, H_KV, T, d_h, s};
    uint64_t acc = 1;
    for (int i = 0; i < 7; ++i) {
        if (f[i] < 0) return UINT64_MAX;
        const uint64_t x = static_cast<uint64_t>(f[i]);
        if (x != 0 && acc > UINT64_MAX / x) return UINT64_MAX;
        acc *= x;
    }
    return acc;
}

extern "C" const char *kvc_status_str(kvc_status s)
{
    switch (s) {
    case KVC_OK: return "ok";
    case KVC_ERR_ARG: return "invalid argument";
    case KVC_ERR_OOM: return "device allocation failed";
    case KVC_ERR_BAD_BLOCK: return "block table entry outside the pool";
    case KVC_ERR_RANGE: return "position or length outside the block table";
    case KVC_ERR_ALIAS: return "two writes to one slot";
    case KVC_ERR_STALE: return "stale block table";
    case KVC_ERR_TIMEOUT: return "device-side wait expired";
    case KVC_ERR_CUDA: return "CUDA runtime error";
    case KVC_ERR_UNSUPPORTED: return "shape not supported by this build";
    }
    return "unknown status";
}

extern "C" uint64_t kvc_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" void kvc_pool_destroy(kvc_pool *pool)
{
    if (!pool) return;
    int prev = -1;
    const bool switched = cudaGetDevice(&prev) == cudaSuccess && prev != pool->device &&
                          cudaSetDevice(pool->device) == cudaSuccess;
    cudaFree(pool->ws);
    cudaFree(pool->base);
    cudaFree(pool->scales);
    cudaFree(pool->absmax);
    cudaFree(pool->err);
    if (switched) cudaSetDevice(prev);
    delete pool;
}

extern "C" kvc_status kvc_pool_create(int64_t num_blocks, int32_t block_size, int32_t num_layers,
                                      int32_t num_kv_heads, int32_t head_dim, kvc_dtype dtype, kvc_pool **out)
{
    if (!out) return KVC_ERR_ARG;
    *out = nullptr;
    if (num_blocks < 1 || block_size < 1 || block_size > 128 || num_layers < 1 || num_kv_heads < 1 ||
        num_kv_heads > 256)
        return KVC_ERR_ARG;
    if (dtype != KVC_BF16 && dtype != KVC_FP8_E4M3 && dtype != KVC_INT4) return KVC_ERR_ARG;
    const int bits = dtype == KVC_BF16 ? 16 : (dtype == KVC_FP8_E4M3 ? 8 : 4);
    const int s = bits / 8;
    // the head widths the attention kernels serve
    const bool dim_ok = dtype == KVC_BF16 ? (head_dim == 64 || head_dim == 128) : head_dim == 128;
    if (!dim_ok) return KVC_ERR_ARG;
    const uint64_t rows = static_cast<uint64_t>(num_layers) * static_cast<uint64_t>(num_blocks) *
                          static_cast<uint64_t>(num_kv_heads) * 2u * static_cast<uint64_t>(block_size);
    if (rows >= (1ull << 31)) return KVC_ERR_ARG;
    const uint64_t pool_bytes = rows * static_cast<uint64_t>(head_dim) * bits / 8;

    kvc_pool *pool = new (std::nothrow) kvc_pool();
    if (!pool) return KVC_ERR_OOM;
    pool->N = num_blocks;
    pool->bs = block_size;
    pool->L = num_layers;
    pool->H_KV = num_kv_heads;
    pool->D = head_dim;
    pool->dtype = dtype;
    pool->s = s;
    pool->bits = bits;
    pool->layer_bytes = pool_bytes / num_layers;
    pool->pool_bytes = pool_bytes;
    if (cudaGetDevice(&pool->device) != cudaSuccess ||
        cudaDeviceGetAttribute(&pool->num_sms, cudaDevAttrMultiProcessorCount, pool->device) != cudaSuccess) {
        delete pool;
        return KVC_ERR_CUDA;
    }
    kvc_status st = KVC_OK;
    if (cudaMalloc(&pool->base, pool_bytes) != cudaSuccess || cudaMalloc(&pool->err, sizeof(uint32_t)) != cudaSuccess ||
        cudaMemset(pool->err, 0, sizeof(uint32_t)) != cudaSuccess)
        st = KVC_ERR_OOM;
    const int nsc = num_layers * 2 * num_kv_heads * head_dim;
    if (st == KVC_OK && dtype != KVC_BF16) {
        if (cudaMalloc(&pool->scales, sizeof(float) * nsc) != cudaSuccess ||
            cudaMalloc(&pool->absmax, sizeof(float) * nsc) != cudaSuccess ||
            cudaMemset(pool->absmax, 0, sizeof(float) * nsc) != cudaSuccess)
            st = KVC_ERR_OOM;
        else {
            fill_kernel<<<(nsc + 255) / 256, 256>>>(pool->scales, 1.f, nsc);
            if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) st = KVC_ERR_CUDA;
            g_launches.fetch_add(1, std::memory_order_relaxed);
        }
    }
    if (st != KVC_OK) {
        (void)cudaGetLastError();
        kvc_pool_destroy(pool);
        return st;
    }
    // Tensor map: the pool as rows of D elements; a box is one 128-byte
    // column band of one block's 2*bs key+value rows, with 128-byte swizzle.
    // int4 rows are 64 bytes: the map's rows are 128-byte lines (two token
    // rows) and a box is one block-head's bs lines.
    pool->tmap_ok = false;
    if (PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder()) {
        const bool lines = bits == 4;
        cuuint64_t gdim[2] = {lines ? 128u : static_cast<cuuint64_t>(head_dim),
                              lines ? static_cast<cuuint64_t>(pool_bytes / 128) : static_cast<cuuint64_t>(rows)};
        cuuint64_t gstride[1] = {lines ? 128u : static_cast<cuuint64_t>(head_dim) * s};
        cuuint32_t box[2] = {lines ? 128u : static_cast<cuuint32_t>(128 / s),
                             static_cast<cuuint32_t>(lines ? block_size : 2 * block_size)};
        cuuint32_t estride[2] = {1, 1};
        const CUresult r = enc(&pool->tmap, bits == 16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                               2, pool->base, gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        pool->tmap_ok = (r == CUDA_SUCCESS);
        // keys and values of 16 positions as separate boxes (the tensor-memory kernels stage
        // them in separate regions); 16-bit pools whose blocks hold whole 16-position groups
        pool->tmap16_ok = false;
        if (bits == 16 && block_size % 16 == 0) {
            cuuint32_t box16[2] = {static_cast<cuuint32_t>(128 / s), 16u};
            const CUresult r16 = enc(&pool->tmap16, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pool->base, gdim, gstride,
                                     box16, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            pool->tmap16_ok = (r16 == CUDA_SUCCESS);
        }
    }
    noalloc_prepare(pool->device);   // the allocation-free decode's scratch: reserved now, not mid-step
    (void)cudaGetLastError();
    *out = pool;
    return KVC_OK;
}

extern "C" kvc_status kvc_pool_info(const kvc_pool *pool, kvc_pool_desc *d)
{
    if (!pool || !d) return KVC_ERR_ARG;
    std::memset(d, 0, sizeof(*d));
    d->layout_version = 1;
    d->block_size = pool->bs;
    d->num_layers = pool->L;
    d->num_kv_heads = pool->H_KV;
    d->head_dim = pool->D;
    d->dtype = pool->dtype;
    d->elem_bytes = pool->s;
    d->elem_bits = pool->bits;
    d->device = pool->device;
    d->num_blocks = pool->N;
    d->block_bytes_per_layer = 2ull * pool->H_KV * pool->bs * pool->D * pool->bits / 8;
    d->layer_bytes = pool->layer_bytes;
    d->bytes_per_token = 2ull * pool->L * pool->H_KV * pool->D * pool->bits / 8;
    d->capacity_tokens = static_cast<uint64_t>(pool->N) * pool->bs;
    d->pool_bytes = pool->pool_bytes;
    d->base = pool->base;
    d->scales = pool->scales;
    return KVC_OK;
}

extern "C" kvc_status kvc_pool_set_scales(kvc_pool *pool, int32_t layer, const float *s_k, const float *s_v,
                                          kvc_stream_t stream)
{
    if (!pool || !s_k || !s_v || pool->dtype == KVC_BF16 || layer < 0 || layer >= pool->L) return KVC_ERR_ARG;
    kvc_status st = check_device(pool);
    if (st != KVC_OK) return st;
    const size_t n = static_cast<size_t>(pool->H_KV) * pool->D;
    float *dst = pool->scales + static_cast<size_t>(layer) * 2 * n;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(dst, s_k, n * sizeof(float), cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaMemcpyAsync(dst + n, s_v, n * sizeof(float), cudaMemcpyDeviceToDevice, s);
    return cuda_status(e);
}

extern "C" kvc_status kvc_calibrate_scales(kvc_pool *pool, int32_t layer, const void *k, const void *v,
                                           int64_t n_tokens, int32_t accumulate, kvc_stream_t stream)
{
    if (!pool || pool->dtype == KVC_BF16 || layer < 0 || layer >= pool->L || n_tokens < 0) return KVC_ERR_ARG;
    if (n_tokens > 0 && (!k || !v || !aligned(k, 2) || !aligned(v, 2))) return KVC_ERR_ARG;
    kvc_status st = check_device(pool);
    if (st != KVC_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int HD = pool->H_KV * pool->D;
    float *amax = pool->absmax + static_cast<size_t>(layer) * 2 * HD;
    cudaError_t e = cudaSuccess;
    if (!accumulate) e = cudaMemsetAsync(amax, 0, sizeof(float) * 2 * HD, s);
    if (e != cudaSuccess) return cuda_status(e);
    if (n_tokens > 0) {
        const int tpc = 64;
        const int64_t gx = (n_tokens + tpc - 1) / tpc;
        if (gx > 0x7FFFFFFF) return KVC_ERR_ARG;
        const int gy = (HD + 255) / 256;
        for (int kv = 0; kv < 2; ++kv) {
            absmax_kernel<<<dim3(static_cast<unsigned>(gx), gy), 256, 0, s>>>(
                static_cast<const uint16_t *>(kv ? v : k), n_tokens, HD, tpc, amax + kv * HD);
            if ((e = cudaGetLastError()) != cudaSuccess) return cuda_status(e);
            g_launches.fetch_add(1, std::memory_order_relaxed);
        }
    }
    scales_from_absmax_kernel<<<(2 * HD + 255) / 256, 256, 0, s>>>(
        amax, pool->scales + static_cast<size_t>(layer) * 2 * HD, 2 * HD, pool->dtype == KVC_INT4 ? 7.f : 448.f);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_status(e);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return KVC_OK;
}

extern "C" kvc_status kvc_calibrate_fp8(kvc_pool *pool, int32_t layer, const void *k, const void *v,
                                        int64_t n_tokens, int32_t accumulate, kvc_stream_t stream)
{
    return kvc_calibrate_scales(pool, layer, k, v, n_tokens, accumulate, stream);
}

extern "C" kvc_status kvc_append(kvc_pool *pool, int32_t layer, const int32_t *block_tables, int32_t max_blocks,
                                 const int32_t *seq_lens, int32_t B, const void *k_new, const void *v_new,
                                 kvc_stream_t stream)
{
    return scatter(pool, layer, block_tables, max_blocks, seq_lens, nullptr, B, 1, k_new, v_new,
                   static_cast<cudaStream_t>(stream));
}

extern "C" kvc_status kvc_write_tokens(kvc_pool *pool, int32_t layer, const int32_t *block_tables, int32_t max_blocks,
                                       const int32_t *start_pos, const int32_t *cu_tokens, int32_t B,
                                       int32_t max_tokens, const void *k, const void *v, kvc_stream_t stream)
{
    if (B > 0 && (!cu_tokens || !aligned(cu_tokens, 4))) return KVC_ERR_ARG;
    return scatter(pool, layer, block_tables, max_blocks, start_pos, cu_tokens, B, max_tokens, k, v,
                   static_cast<cudaStream_t>(stream));
}

extern "C" kvc_status kvc_pool_sync_status(kvc_pool *pool, kvc_stream_t stream)
{
    if (!pool) return KVC_ERR_ARG;
    kvc_status st = check_device(pool);
    if (st != KVC_OK) return st;
    uint32_t bits = 0;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess ||
        cudaMemcpy(&bits, pool->err, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(pool->err, 0, sizeof(bits)) != cudaSuccess)
        return KVC_ERR_CUDA;
    if ((bits & KVC_EBIT_TIMEOUT) && pool->ws) {
        // an expired wait may have left split arrival counters short of their count: restart them at zero
        if (cudaMemset(pool->ws, 0, pool->ws_counters * sizeof(uint32_t)) != cudaSuccess) return KVC_ERR_CUDA;
    }
    if (bits & KVC_EBIT_BAD_BLOCK) return KVC_ERR_BAD_BLOCK;
    if (bits & KVC_EBIT_RANGE) return KVC_ERR_RANGE;
    if (bits & KVC_EBIT_TIMEOUT) return KVC_ERR_TIMEOUT;
    return KVC_OK;
}
