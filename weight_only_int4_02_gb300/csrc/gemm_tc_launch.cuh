// Host-side launch and set-up of w4a16_tc_kernel<TM, KSUB>; included by one .cu file per tile shape.
#pragma once
#include "gemm_tc.cuh"

namespace w4a16 {

template <int TM, int KSUB>
cudaError_t setup_tc()
{
    return cudaFuncSetAttribute(w4a16_tc_kernel<TM, KSUB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TcCfg<TM, KSUB>::kSmemBytes);
}

template <int TM, int KSUB>
cudaError_t launch_tc(const CUtensorMap& tmap, const GemmParams& p, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(TcCfg<TM, KSUB>::kThreads);
    cfg.dynamicSmemBytes = TcCfg<TM, KSUB>::kSmemBytes;
    cfg.stream = stream;
    // Programmatic dependent launch: the next kernel may start its prologue and
    // weight stream while this one drains; it waits for this one before reading X.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, w4a16_tc_kernel<TM, KSUB>, tmap, p);
}

}  // namespace w4a16

#define W4A16_INSTANTIATE_TC(TM, KSUB)                                                              \
    namespace w4a16 {                                                                               \
    template cudaError_t setup_tc<TM, KSUB>();                                                      \
    template cudaError_t launch_tc<TM, KSUB>(const CUtensorMap&, const GemmParams&, cudaStream_t);  \
    }
