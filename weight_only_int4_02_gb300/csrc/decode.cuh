// Parameters and launch of the decode kernel (decode.cu): the W4A16 matmul for up
// to sixteen rows of X with the register-level unpack feeding warp-level MMAs,
// column blocks of 16 to 128 output features, each processed by one CTA over the
// whole reduction dimension, weights, scales and X staged by TMA.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4a16 {

constexpr int kDecThreads = 320;    // 8 consumer warps, 1 weight producer warp, 1 X producer warp
constexpr int kDecStageRows = 16;   // rows of 32 values of k per pipeline stage (512 values)

struct DecodeParams {
    __half* y;               // [M][N]
    const __half* bias;      // [N] or null (fused epilogue)
    const __half* residual;  // [M][ldr] or null (may be y itself)
    int* status;             // error word: bit 0 = a wait timed out
    long long wait_limit_ns;
    int act;                 // 0 none, 1 SiLU, 2 ReLU
    int ldy, ldr;            // row strides (elements) of y and the residual: >= N
    int M, N, ng;
    int g_shift;             // log2(G) for G a power of two; 30 for one group
    int tile_rows;           // rows of 32 k per column tile in the packed layout: 2 * KC
    int rows;                // rows that hold data: K / 32 (K is a multiple of 32)
    int stages;              // ceil(rows / kDecStageRows)
    int scale_rows;          // group rows the scale map's box brings per stage
    int x_rows;              // rows of X the X map's box brings per row of k: M (<= mr)
    int ring;                // pipeline slots (2 .. kDecMaxRing)
};

constexpr int kDecMaxRing = 16;
constexpr int kDecSmemBudget = 104 * 1024;   // the ring; two CTAs share an SM
// Packed bytes the ring holds (fewer where the budget says so), by block width, as
// measured on GB300 for launches chained back to back: 24 KB (six stages) for blocks
// of 16 columns, whose deeper rings ran slower, 80 KB (four stages) for 80 columns,
// 64 KB for the others.
constexpr int decode_words_in_flight(int cb) { return cb == 16 ? 24 * 1024 : cb == 80 ? 80 * 1024 : 64 * 1024; }

// Shared-memory bytes of one pipeline slot, and of a launch with `ring` slots
// (ring * slot <= kDecSmemBudget).
constexpr int decode_slot_bytes(int cb, int x_rows) { return kDecStageRows * (cb * 16 + cb * 2 + x_rows * 64); }
constexpr int decode_smem_bytes(int cb, int x_rows, int ring)
{
    return ring * decode_slot_bytes(cb, x_rows) + 3 * kDecMaxRing * 8 + 16 + 128;
}

// Tensor maps (built on the host):
//   tmap_w: the packed words as uint32 [n_tiles * tile_rows][512], box {box * 4, 16};
//   tmap_s: the tile-ordered scales as 16-bit [n_tiles * ng][128], box {cb, scale_rows}
//           (box {16, scale_rows} for cb 48 and 80);
//   box = 16 for cb 48 and 80 (blocks that can straddle two tiles), else min(cb, 64);
//   tmap_x: X as 16-bit {32, M, K / 32} with strides {2 ldx, 64} bytes, box {32, M, 16},
//           so a stage lands as [16 rows of k][M rows of X][32 values].
// mr: 8 or 16 (rows of X the kernel is built for, >= M); cb: 16, 32, 64 or 128, and 48 or
// 80 with mr = 8; grid = ceil(N / cb);
// the dynamic shared memory is decode_smem_bytes(cb, M, p.ring).
cudaError_t launch_decode(const CUtensorMap& tmap_w, const CUtensorMap& tmap_s, const CUtensorMap& tmap_x,
                          const DecodeParams& p, int mr, int cb, bool epi, int grid, cudaStream_t stream);

// Shared-memory attributes of every instantiation (once per device).
cudaError_t setup_decode();

}  // namespace w4a16
