// Instances of the tensor-memory (tcgen05) decode kernel.
#include "kvc_decode_tc.cuh"

namespace kvc {

template <int G>
static DecodeKernel decode_tc_instance()
{
    static DecodeKernel k = [] {
        DecodeKernel r;
        r.fn = reinterpret_cast<const void *>(&decode_tc_kernel<G>);
        r.smem = kTcSmem;
        r.ctas_per_sm = 0;
        if (cudaFuncSetAttribute(&decode_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, r.smem) ==
            cudaSuccess) {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, &decode_tc_kernel<G>, kTcThreads, r.smem) ==
                cudaSuccess)
                r.ctas_per_sm = n;
        }
        return r;
    }();
    return k;
}

DecodeKernel select_decode_tc(int D, int g, int dtype)
{
    if (D != 128 || dtype != KVC_BF16 || g != 32) return DecodeKernel{nullptr, 0, 0};
    return decode_tc_instance<32>();
}

}  // namespace kvc
