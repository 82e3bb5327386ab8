// Host-side launch and set-up of w4a16_tc_kernel<TM>; included by one .cu file per TM.
#pragma once
#include "gemm_tc.cuh"

namespace w4a16 {

template <int TM>
cudaError_t setup_tc()
{
    return cudaFuncSetAttribute(w4a16_tc_kernel<TM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TcCfg<TM>::kSmemBytes);
}

template <int TM>
cudaError_t launch_tc(const CUtensorMap& tmap, const GemmParams& p, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = TcCfg<TM>::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, w4a16_tc_kernel<TM>, tmap, p);
}

}  // namespace w4a16

#define W4A16_INSTANTIATE_TC(TM)                                                                  \
    namespace w4a16 {                                                                             \
    template cudaError_t setup_tc<TM>();                                                          \
    template cudaError_t launch_tc<TM>(const CUtensorMap&, const GemmParams&, cudaStream_t);      \
    }
