// Instances of the tensor-memory (tcgen05) prefill kernel.
#include "kvc_prefill_tc.cuh"

namespace kvc {

template <int D>
static DecodeKernel prefill_tc_instance()
{
    static DecodeKernel k = [] {
        DecodeKernel r;
        r.fn = reinterpret_cast<const void *>(&prefill_tc_kernel<D>);
        r.smem = PrefillTcCfg<D>::SMEM;
        r.ctas_per_sm = 0;
        if (cudaFuncSetAttribute(&prefill_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, r.smem) ==
            cudaSuccess) {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, &prefill_tc_kernel<D>, kPtThreads, r.smem) ==
                cudaSuccess)
                r.ctas_per_sm = n;
        }
        return r;
    }();
    return k;
}

DecodeKernel select_prefill_tc(int D, int dtype)
{
    if (dtype != KVC_BF16) return DecodeKernel{nullptr, 0, 0};
    if (D == 64) return prefill_tc_instance<64>();
    if (D == 128) return prefill_tc_instance<128>();
    return DecodeKernel{nullptr, 0, 0};
}

}  // namespace kvc
