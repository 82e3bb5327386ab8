// Host-side launch and set-up of w4a16_tc_kernel<TM, KSUB, EPI, FMT>; included by one .cu file per tile shape
// and weight format.
#pragma once
#include "gemm_tc.cuh"

namespace w4a16 {

// Dynamic shared memory of the instantiation.
template <int TM, int KSUB, bool EPI, int FMT>
cudaError_t setup_tc()
{
    using C = TcCfg<TM, KSUB, FMT>;
    return cudaFuncSetAttribute(w4a16_tc_kernel<TM, KSUB, EPI, FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                C::kSmemBytes);
}

template <int TM, int KSUB, bool EPI, int FMT>
cudaError_t launch_tc(const CUtensorMap& tmap, const GemmParams& p, cudaStream_t stream)
{
    using C = TcCfg<TM, KSUB, FMT>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.grid);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    // Programmatic dependent launch: the next kernel may start its prologue and
    // weight stream while this one drains; it waits for this one before reading X.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, w4a16_tc_kernel<TM, KSUB, EPI, FMT>, tmap, p);
}

}  // namespace w4a16

// Both epilogue variants of one tile shape and weight format (w4a16::kFmt*).
#define W4A16_INSTANTIATE_TC(TM, KSUB, FMT)                                                                   \
    namespace w4a16 {                                                                                         \
    template cudaError_t setup_tc<TM, KSUB, false, FMT>();                                                    \
    template cudaError_t setup_tc<TM, KSUB, true, FMT>();                                                     \
    template cudaError_t launch_tc<TM, KSUB, false, FMT>(const CUtensorMap&, const GemmParams&, cudaStream_t); \
    template cudaError_t launch_tc<TM, KSUB, true, FMT>(const CUtensorMap&, const GemmParams&, cudaStream_t);  \
    }
