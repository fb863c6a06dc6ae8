// Decode attention that allocates nothing: the split-K partials live in a
// fixed, file-scope device array instead of the pool's cudaMalloc'd workspace.
//
// Some callers may not allocate device memory in the middle of a decode step:
// a serving loop whose device memory is entirely pre-reserved by its own
// caching allocator (a cudaMalloc there fails, or fragments memory the engine
// has promised to KV blocks), and latency-critical loops where cudaMalloc /
// cudaFree would synchronise the device and stall every other stream.  For
// them, kvc_decode_attn_noalloc runs the same kernels as kvc_decode_attn with
// partials in kvc_noalloc_scratch.
#include <cmath>
#include <mutex>
#include <unordered_map>

#include "kvc_decode_tc.cuh"

namespace kvc {

// 8 MiB per device, held by every GPU that loads the library until the process exits.
constexpr size_t kNoallocScratchFloats = size_t(2) << 20;
static __device__ __align__(256) float kvc_noalloc_scratch[kNoallocScratchFloats];

// Device address of the scratch array in the calling thread's current context.
// In host code the array's name is only a host-side stand-in, so the address
// comes from cudaGetSymbolAddress, made with the pool's device current.  It is
// looked up once per context and cached under the context's unique id: after a
// device reset the runtime creates a new primary context (a new id), the module
// is loaded again and the array may sit elsewhere, so the stale address of the
// old context is never used.  Without the driver's context-id entry points the
// address is looked up on every call.
using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

template <class Fn>
static Fn driver_fn(const char *name)
{
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return reinterpret_cast<Fn>(f);
}

static float *lookup_scratch()
{
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, kvc_noalloc_scratch) != cudaSuccess) {
        (void)cudaGetLastError();
        return nullptr;
    }
    return static_cast<float *>(p);
}

static float *noalloc_scratch_ptr(int device)
{
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    static std::mutex mu;
    static std::unordered_map<unsigned long long, float *> by_context;
    if (cudaSetDevice(device) != cudaSuccess) return nullptr;   // makes the device's primary context current
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
        return lookup_scratch();
    std::lock_guard<std::mutex> lock(mu);
    auto it = by_context.find(id);
    if (it != by_context.end()) return it->second;
    float *p = lookup_scratch();
    if (p) by_context.emplace(id, p);
    return p;
}

static bool is_aligned(const void *ptr, size_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

// Called by kvc_pool_create with the pool's device current: loads the module and
// reserves the array there (and caches its address) when the pool is created,
// not in the middle of a later decode step.
void noalloc_prepare(int device) { (void)noalloc_scratch_ptr(device); }

}  // namespace kvc

using namespace kvc;

extern "C" kvc_status kvc_decode_attn_noalloc(kvc_pool *pool, int32_t layer, const void *q, int32_t num_q_heads,
                                              const int32_t *block_tables, int32_t max_blocks,
                                              const int32_t *seq_lens, int32_t B, float *out, float *lse,
                                              float scale, kvc_stream_t stream)
{
    if (B < 0 || B > 65535) return KVC_ERR_ARG;
    if (B == 0) return pool ? KVC_OK : KVC_ERR_ARG;
    if (!pool || !q || !block_tables || !seq_lens || !out) return KVC_ERR_ARG;
    if (layer < 0 || layer >= pool->L) return KVC_ERR_ARG;
    if (num_q_heads <= 0 || num_q_heads % pool->H_KV != 0) return KVC_ERR_ARG;
    if (num_q_heads / pool->H_KV > 32) return KVC_ERR_UNSUPPORTED;
    if (pool->bs != kBS || !pool->tmap_ok) return KVC_ERR_UNSUPPORTED;
    if (max_blocks <= 0 || max_blocks > (1 << 26) || !std::isfinite(scale)) return KVC_ERR_ARG;
    if (!is_aligned(q, 16) || !is_aligned(out, 16) || (lse && !is_aligned(lse, 4)) || !is_aligned(block_tables, 4) ||
        !is_aligned(seq_lens, 4))
        return KVC_ERR_ARG;
    kvc_status st = check_device(pool);
    if (st != KVC_OK) return st;
    float *scratch = noalloc_scratch_ptr(pool->device);   // cached per context; looked up at pool creation
    if (!scratch) return KVC_ERR_CUDA;

    DecodeParams p{};
    p.q = static_cast<const uint16_t *>(q);
    p.bt = block_tables;
    p.lens = seq_lens;
    p.bt_stride = max_blocks;
    p.max_blocks = max_blocks;
    p.len_base = 0;
    p.B = B;
    p.ppu = 1;
    p.n_pos = B;
    p.H_Q = num_q_heads;
    p.H_KV = pool->H_KV;
    p.g = num_q_heads / pool->H_KV;
    p.layer = layer;
    p.N = pool->N;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.s_k = pool->scales ? pool->scales + static_cast<size_t>(layer) * 2 * pool->H_KV * pool->D : nullptr;
    p.s_v = p.s_k ? p.s_k + static_cast<size_t>(pool->H_KV) * pool->D : nullptr;
    p.out = out;
    p.lse = lse;
    p.err = pool->err;

    const DecodeKernel tc = tc_kernel_for(pool, p);   // the kernel kvc_decode_attn would launch
    const DecodeKernel k =
        tc.fn                       ? tc
        : pool->dtype == KVC_FP8_E4M3 ? select_decode_fp8(pool->D, p.g)
        : pool->dtype == KVC_INT4   ? select_decode_int4(pool->D, p.g)
                                    : select_decode_bf16(pool->D, p.g);
    if (!k.fn) return KVC_ERR_UNSUPPORTED;
    if (k.ctas_per_sm <= 0) return KVC_ERR_CUDA;
    if (tc.fn)
        choose_split_tc(pool, p.B * p.H_KV, p.max_blocks, k.ctas_per_sm, k.split_unit, &p.chunk, &p.max_splits);
    else choose_split(pool, p.B * p.H_KV, p.max_blocks, k.ctas_per_sm, &p.chunk, &p.max_splits, n_tiles(p.g));
    if (p.max_splits > 65535) return KVC_ERR_UNSUPPORTED;
    if (p.max_splits > 1) {
        // partials: o [B][H_Q][splits][D] then (max, sum) [B][H_Q][splits]; every slot read is written first
        const size_t n = static_cast<size_t>(p.B) * p.H_Q * p.max_splits;
        if (n * (static_cast<size_t>(pool->D) + 2) > kNoallocScratchFloats) return KVC_ERR_ARG;
        p.part_o = scratch;
        p.part_ml = reinterpret_cast<float2 *>(scratch + n * pool->D);
    }
    const dim3 grid(p.max_splits, p.H_KV, p.B);
    void *args[] = {const_cast<CUtensorMap *>(k.tmap16 ? &pool->tmap16 : &pool->tmap), &p};
    const cudaError_t e = cudaLaunchKernel(k.fn, grid, dim3(k.threads), args, k.smem,
                                           static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_status(e);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (p.max_splits > 1) return launch_split_merge(p, pool->D, static_cast<cudaStream_t>(stream));
    return KVC_OK;
}
