// e4m3-pool instances of the decode-attention kernel.
#include "kvc_decode.cuh"

namespace kvc {

kvc_status launch_decode_fp8(const kvc_pool *pool, DecodeParams &p, cudaStream_t stream)
{
    const int NT = n_tiles(p.ppu * p.g);
    if (pool->D != 128) return KVC_ERR_UNSUPPORTED;
    if (!p.lens) return run_decode(pool, p, decode_instance<128, 4, KV_E4M3, false, true>(), stream);
    {   // the balanced persistent kernel where the batch suits it
        const DecodeKernel kp = NT == 1 ? persistent_instance<128, 1, KV_E4M3, false>()
                              : NT == 2 ? persistent_instance<128, 2, KV_E4M3, false>()
                                        : DecodeKernel{nullptr, 0, 0};   // 32-column groups keep the split kernel
        const kvc_status st = run_decode_persistent(const_cast<kvc_pool *>(pool), p, kp, stream);
        if (st != KVC_ERR_UNSUPPORTED) return st;
    }
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
