// int4-pool instances of the decode-attention kernel.
#include "kvc_prefill.cuh"

namespace kvc {

DecodeKernel select_decode_int4(int D, int g)
{
    const int NT = n_tiles(g);
    if (D != 128) return DecodeKernel{nullptr, 0, 0};
    return NT == 1 ? decode_instance<128, 1, KV_INT4, false>()
         : NT == 2 ? decode_instance<128, 2, KV_INT4, false>()
                   : decode_instance<128, 4, KV_INT4, false>();
}

kvc_status launch_decode_int4(const kvc_pool *pool, DecodeParams &p, cudaStream_t stream)
{
    if (pool->D != 128) return KVC_ERR_UNSUPPORTED;
    const DecodeKernel k = p.lens ? select_decode_int4(pool->D, p.ppu * p.g)
                                  : decode_instance<128, 4, KV_INT4, false, true>();   // prefill tiles
    if (!k.fn) return KVC_ERR_UNSUPPORTED;
    return run_decode(pool, p, k, stream);
}

}  // namespace kvc

namespace kvc {

// The mixed decode + prefill kernel for an int4 pool: d_h 128, decode groups of up to 16 query heads.
DecodeKernel select_mixed_int4(int D, int g)
{
    const int NT = n_tiles(g);
    if (D != 128 || NT > 2) return DecodeKernel{nullptr, 0, 0};
    return NT == 1 ? mixed_instance<128, 1, KV_INT4, false, false>() : mixed_instance<128, 2, KV_INT4, false, false>();
}

}  // namespace kvc
