// bf16-pool instances of the decode-attention kernel.
#include <cstdlib>

#include "kvc_decode.cuh"

namespace kvc {

template <int D>
static DecodeKernel pick_bf16(int NT, bool psplit)
{
    if (NT == 1) return psplit ? decode_instance<D, 1, false, true>() : decode_instance<D, 1, false, false>();
    if (NT == 2) return psplit ? decode_instance<D, 2, false, true>() : decode_instance<D, 2, false, false>();
    return psplit ? decode_instance<D, 4, false, true>() : decode_instance<D, 4, false, false>();
}

kvc_status launch_decode_bf16(const kvc_pool *pool, DecodeParams &p, cudaStream_t stream)
{
    // KVC_PSPLIT=0 feeds the softmax weights to the value mixture as one bf16
    // operand instead of a high/low pair (faster, ~8 fewer bits per weight).
    static const bool psplit = [] {
        const char *e = std::getenv("KVC_PSPLIT");
        return !(e && e[0] == '0');
    }();
    const int NT = n_tiles(p.ppu * p.g);
    DecodeKernel k;
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
    const char *e = std::getenv("KVC_PSPLIT");
    const bool psplit = !(e && e[0] == '0');
    const int NT = g <= 8 ? 1 : (g <= 16 ? 2 : 4);
    if (D == 64) return pick_bf16<64>(NT, psplit);
    if (D == 128) return pick_bf16<128>(NT, psplit);
    return DecodeKernel{nullptr, 0, 0};
}

}  // namespace kvc
