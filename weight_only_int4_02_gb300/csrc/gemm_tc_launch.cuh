// Host-side launch and set-up of w4a16_tc_kernel<TM, KSUB, CL, EPI, ZP>; included by one .cu file per tile
// shape and weight format (zero-point 8, or per-group zero-points).
#pragma once
#include "gemm_tc.cuh"

namespace w4a16 {

// Dynamic shared memory, and for clusters the number of clusters the device can
// hold at once (0 when the query fails).
template <int TM, int KSUB, int CL, bool EPI, bool ZP>
cudaError_t setup_tc(int* max_clusters)
{
    using C = TcCfg<TM, KSUB, ZP>;
    auto kernel = w4a16_tc_kernel<TM, KSUB, CL, EPI, ZP>;
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

template <int TM, int KSUB, int CL, bool EPI, bool ZP>
cudaError_t launch_tc(const CUtensorMap& tmap, const GemmParams& p, cudaStream_t stream)
{
    using C = TcCfg<TM, KSUB, ZP>;
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
    return cudaLaunchKernelEx(&cfg, w4a16_tc_kernel<TM, KSUB, CL, EPI, ZP>, tmap, p);
}

}  // namespace w4a16

// Both epilogue variants of one tile shape and weight format (ZP = per-group zero-points).
#define W4A16_INSTANTIATE_TC(TM, KSUB, CL, ZP)                                                                    \
    namespace w4a16 {                                                                                             \
    template cudaError_t setup_tc<TM, KSUB, CL, false, ZP>(int*);                                                 \
    template cudaError_t setup_tc<TM, KSUB, CL, true, ZP>(int*);                                                  \
    template cudaError_t launch_tc<TM, KSUB, CL, false, ZP>(const CUtensorMap&, const GemmParams&, cudaStream_t); \
    template cudaError_t launch_tc<TM, KSUB, CL, true, ZP>(const CUtensorMap&, const GemmParams&, cudaStream_t);  \
    }
