// Instances of the tensor-memory (tcgen05) decode kernels (bf16 pools; e4m3 pools in kvc_decode_tc8.cu).
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
        r.threads = kTcThreads;
        r.tmap16 = true;
        r.split_unit = kTcBlocks;   // whole tiles
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
    if (D != 128 || g != 32) return DecodeKernel{nullptr, 0, 0};
    if (dtype == KVC_BF16) return decode_tc_instance<32>();
    if (dtype == KVC_FP8_E4M3) return select_decode_tc8(D, g);
    return DecodeKernel{nullptr, 0, 0};
}

}  // namespace kvc
