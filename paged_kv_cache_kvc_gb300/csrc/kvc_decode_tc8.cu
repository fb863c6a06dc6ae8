// Instances of the tensor-memory (tcgen05) decode kernel for e4m3 pools.
#include "kvc_decode_tc8.cuh"

namespace kvc {

template <int G>
static DecodeKernel decode_tc8_instance()
{
    static DecodeKernel k = [] {
        DecodeKernel r;
        r.fn = reinterpret_cast<const void *>(&decode_tc8_kernel<G>);
        r.smem = kT8Smem;
        r.ctas_per_sm = 0;
        r.threads = kT8Threads;
        r.tmap16 = false;   // boxes of whole blocks (keys and values, 32 rows of 128 codes)
        r.split_unit = 1;   // even shares of the blocks
        if (cudaFuncSetAttribute(&decode_tc8_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, r.smem) ==
            cudaSuccess) {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, &decode_tc8_kernel<G>, kT8Threads, r.smem) ==
                cudaSuccess)
                r.ctas_per_sm = n;
        }
        return r;
    }();
    return k;
}

DecodeKernel select_decode_tc8(int D, int g)
{
    if (D != 128 || g != 32) return DecodeKernel{nullptr, 0, 0};
    return decode_tc8_instance<32>();
}

}  // namespace kvc
