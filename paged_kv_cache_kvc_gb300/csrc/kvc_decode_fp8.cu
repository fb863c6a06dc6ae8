// e4m3-pool instances of the decode-attention kernel.
#include "kvc_prefill.cuh"

namespace kvc {

kvc_status launch_decode_fp8(const kvc_pool *pool, DecodeParams &p, cudaStream_t stream)
{
    const int NT = n_tiles(p.ppu * p.g);
    if (pool->D != 128) return KVC_ERR_UNSUPPORTED;
    if (!p.lens) return run_decode(pool, p, decode_instance<128, 4, KV_E4M3, false, true>(), stream);
    DecodeKernel k = NT == 1 ? decode_instance<128, 1, KV_E4M3, false>()
                   : NT == 2 ? decode_instance<128, 2, KV_E4M3, false>()
                             : decode_instance<128, 4, KV_E4M3, false>();
    return run_decode(pool, p, k, stream);
}

}  // namespace kvc

namespace kvc {

// The e4m3 kernel instance kvc_decode_attn would launch for head width D and group size g.
DecodeKernel select_decode_fp8(int D, int g)
{
    const int NT = g <= 8 ? 1 : (g <= 16 ? 2 : 4);
    if (D != 128) return DecodeKernel{nullptr, 0, 0};
    return NT == 1 ? decode_instance<128, 1, KV_E4M3, false>()
         : NT == 2 ? decode_instance<128, 2, KV_E4M3, false>()
                   : decode_instance<128, 4, KV_E4M3, false>();
}

}  // namespace kvc

namespace kvc {

// The mixed decode + prefill kernel for an e4m3 pool: d_h 128, decode groups of up to 16 query heads.
DecodeKernel select_mixed_fp8(int D, int g)
{
    const int NT = n_tiles(g);
    if (D != 128 || NT > 2) return DecodeKernel{nullptr, 0, 0};
    return NT == 1 ? mixed_instance<128, 1, KV_E4M3, false, false>() : mixed_instance<128, 2, KV_E4M3, false, false>();
}

}  // namespace kvc
