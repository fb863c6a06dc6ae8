// bf16-pool instances of the decode-attention kernel.
#include <cstdlib>

#include "kvc_prefill.cuh"

namespace kvc {

template <int D>
static DecodeKernel pick_bf16(int NT, bool psplit)
{
    if (NT == 1) return psplit ? decode_instance<D, 1, KV_BF16, true>() : decode_instance<D, 1, KV_BF16, false>();
    if (NT == 2) return psplit ? decode_instance<D, 2, KV_BF16, true>() : decode_instance<D, 2, KV_BF16, false>();
    return psplit ? decode_instance<D, 4, KV_BF16, true>() : decode_instance<D, 4, KV_BF16, false>();
}

kvc_status launch_decode_bf16(const kvc_pool *pool, DecodeParams &p, cudaStream_t stream)
{
    // The softmax weights enter the value mixture as a bf16 high/low pair for up
    // to 16 query columns; 32-column units (MQA, prefill tiles) take one bf16
    // operand so their registers fit.  KVC_PSPLIT=0 / 1 forces either.
    const int NT = n_tiles(p.ppu * p.g);
    const char *e = std::getenv("KVC_PSPLIT");
    const bool psplit = e ? e[0] != '0' : NT <= 2;
    DecodeKernel k;
    if (!p.lens) {   // prefill tiles: per-column causal lengths, 32 columns
        if (pool->D == 64) k = decode_instance<64, 4, KV_BF16, false, true>();
        else if (pool->D == 128) k = decode_instance<128, 4, KV_BF16, false, true>();
        else return KVC_ERR_UNSUPPORTED;
        return run_decode(pool, p, k, stream);
    }
    switch (pool->D) {
    case 64: k = pick_bf16<64>(NT, psplit); break;
    case 128: k = pick_bf16<128>(NT, psplit); break;
    default: return KVC_ERR_UNSUPPORTED;
    }
    return run_decode(pool, p, k, stream);
}

}  // namespace kvc

namespace kvc {

// The bf16 kernel instance kvc_decode_attn would launch for head width D and group size g.
DecodeKernel select_decode_bf16(int D, int g)
{
    const int NT = n_tiles(g);
    const char *e = std::getenv("KVC_PSPLIT");
    const bool psplit = e ? e[0] != '0' : NT <= 2;
    if (D == 64) return pick_bf16<64>(NT, psplit);
    if (D == 128) return pick_bf16<128>(NT, psplit);
    return DecodeKernel{nullptr, 0, 0};
}

}  // namespace kvc

namespace kvc {

// The mixed decode + prefill kernel for a bf16 pool: decode groups of up to 16 query heads;
// fast_prefill (groups of at most 4) takes the query-tiled prefill.
DecodeKernel select_mixed_bf16(int D, int g, bool fast_prefill)
{
    const int NT = n_tiles(g);
    if (NT > 2 || (fast_prefill && g > 4)) return DecodeKernel{nullptr, 0, 0};
    const bool fast = fast_prefill;
    if (D == 64)
        return NT == 2 ? mixed_instance<64, 2, KV_BF16, true, false>()
             : fast    ? mixed_instance<64, 1, KV_BF16, true, true>() : mixed_instance<64, 1, KV_BF16, true, false>();
    if (D == 128)
        return NT == 2 ? mixed_instance<128, 2, KV_BF16, true, false>()
             : fast    ? mixed_instance<128, 1, KV_BF16, true, true>() : mixed_instance<128, 1, KV_BF16, true, false>();
    return DecodeKernel{nullptr, 0, 0};
}

DecodeKernel select_prefill_bf16(int D, int g)
{
    if (g > 4) return DecodeKernel{nullptr, 0, 0};
    if (D == 64) return prefill_instance<64>();
    if (D == 128) return prefill_instance<128>();
    return DecodeKernel{nullptr, 0, 0};
}

}  // namespace kvc
