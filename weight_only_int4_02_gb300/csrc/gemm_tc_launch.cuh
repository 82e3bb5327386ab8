// Host-side launch and set-up of w4a16_tc_kernel<TM, KSUB, CL, EPI, FMT>; included by one .cu file per tile
// shape and weight format.
#pragma once
#include "gemm_tc.cuh"

namespace w4a16 {

// Dynamic shared memory, and for clusters the number of clusters the device can
// hold at once (0 when the query fails).
template <int TM, int KSUB, int CL, bool EPI, int FMT>
cudaError_t setup_tc(int* max_clusters)
{
    using C = TcCfg<TM, KSUB, FMT>;
    auto kernel = w4a16_tc_kernel<TM, KSUB, CL, EPI, FMT>;
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    *max_clusters = 0;
    if (CL > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * CL);
        cfg.blockDim = dim3(C::kThreads);
        cfg.dynamicSmemBytes = C::kSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = CL;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(max_clusters, kernel, &cfg) != cudaSuccess) {
            *max_clusters = 0;
            cudaGetLastError();
        }
    }
    return cudaSuccess;
}

template <int TM, int KSUB, int CL, bool EPI, int FMT>
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
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int n = 1;
    if (CL > 1) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = CL;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        n = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, w4a16_tc_kernel<TM, KSUB, CL, EPI, FMT>, tmap, p);
}

}  // namespace w4a16

// Both epilogue variants of one tile shape and weight format (w4a16::kFmt*).
#define W4A16_INSTANTIATE_TC(TM, KSUB, CL, FMT)                                                                    \
    namespace w4a16 {                                                                                              \
    template cudaError_t setup_tc<TM, KSUB, CL, false, FMT>(int*);                                                 \
    template cudaError_t setup_tc<TM, KSUB, CL, true, FMT>(int*);                                                  \
    template cudaError_t launch_tc<TM, KSUB, CL, false, FMT>(const CUtensorMap&, const GemmParams&, cudaStream_t); \
    template cudaError_t launch_tc<TM, KSUB, CL, true, FMT>(const CUtensorMap&, const GemmParams&, cudaStream_t);  \
    }
