// Parameters and launch of the CUDA-core W4A16 kernel for one to four rows of X
// (gemv.cu): column blocks of 16 or 32 adjacent output features, each processed
// by one CTA over the whole reduction dimension, the packed words and scales
// streamed by TMA through a shared-memory ring.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4a16 {

constexpr int kGemvThreads = 320;     // 8 consumer warps, 1 producer warp, 1 X converter warp
constexpr int kGemvStageK = 1024;     // values of k per pipeline stage (32 rows of 32)

struct GemvParams {
    const __half* x;         // [M][ldx]
    __half* y;               // [M][ldy]
    const __half* bias;      // [N] or null (fused epilogue)
    const __half* residual;  // [M][ldr] or null (may be y itself)
    int ldx, ldy, ldr;       // row strides (elements): ldx >= K, ldy and ldr >= N
    int* status;             // error word: bit 0 = a wait timed out
    long long wait_limit_ns;
    int act;                 // 0 none, 1 SiLU, 2 ReLU
    int M, N, K, ng;
    int g_shift;             // log2(G) for G a power of two; 30 for one group
    int tile_rows;           // rows of 32 k per column tile in the packed layout: 2 * KC
    int rows;                // rows that hold data: ceil(K / 32)
    int stages;              // stages per block: ceil(rows / 32)
    int scale_rows;          // group rows of scales each stage's copy brings (the scale map's box height)
    int blocks;              // column blocks: ceil(N / cb)
};

// Tensor maps (built on the host): tmap_w views the packed words as uint32
// [n_tiles * tile_rows][512] with a box of {cb * 4, 32}; tmap_s views the scales as
// 16-bit [n_tiles * ng][128] with a box of {cb, scale_rows}.
// mr: 1, 2 or 4 (rows of X the kernel is built for, >= M); cb: 16 or 32 columns per block.
cudaError_t launch_gemv(const CUtensorMap& tmap_w, const CUtensorMap& tmap_s, const GemvParams& p, int mr, int cb,
                        bool epi, int grid, cudaStream_t stream);

// Shared-memory attributes and residency of every instantiation (once per device).
cudaError_t setup_gemv();

// CTAs of the instantiation for (mr, cb, epilogue) that one SM holds at once.
int gemv_resident_ctas(int mr, int cb, bool epi);

}  // namespace w4a16
