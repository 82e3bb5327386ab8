/*
 * w4a16.h — C ABI of libw4a16.so: weight-only INT4 x FP16 matmul on GB300 (sm_103a).
 *
 *   Y[M][N] = X[M][K] (FP16) x dequant(Wq)[K][N],   dequant(Wq)[k][n] = (q[k][n] - 8) * s[k/G][n]
 *
 * accumulated in FP32 and stored as FP16 (round to nearest even).
 *
 * The operation is the one the pages on the Marlin kernel describe:
 *  - "quant_marlin_kernel" (aicassindra.com), "The architecture: every piece
 *    explained": INT4 codes packed eight to a 32-bit word in a kernel-specific
 *    permuted order, one FP16 scale per group of weights along the reduction
 *    dimension (commonly 128), unpack to FP16 and multiply by the group scale,
 *    tensor-core MMA against FP16 activations, split-K with a global reduction
 *    of partial sums; activations stay FP16 and the output is FP16.
 *  - same page, "End-to-end flow": activations (tokens x in-features) times
 *    weights (in-features x out-features); repacking is done once, offline.
 *  - "Low-Precision Quantization Kernels in Production" (llms.blog), section 1
 *    (Marlin, "Pre-Permuted Weight Layouts"): the packed layout is a contract
 *    between the repacking step and the kernel; section 3 (FlashInfer): split-K
 *    with a deterministic reduction in global memory, CUDA Graph capture.
 * The zero-point 8 is the symmetric reading (the pages print no zero-point).
 * w4a16_gemm_zp takes one integer zero-point z[g][n] in 0..15 per group and
 * column instead: dequant(Wq)[k][n] = (q[k][n] - z[k/G][n]) * s[k/G][n], the
 * 4-bit format of AWQ checkpoints, which "Low-Precision Quantization Kernels in
 * Production" (llms.blog), section 1, lists among those the Marlin family serves.
 *
 * Conventions for every entry point:
 *  - Pointers named "device" are CUDA device pointers of the current device,
 *    owned by the caller, and must be 16-byte aligned. Arrays are row-major and
 *    contiguous. FP16 values are passed as IEEE binary16 bit patterns (uint16_t).
 *  - Work is enqueued on `stream` (NULL = the legacy default stream) and the
 *    call returns without synchronising. Results are ready when the stream is.
 *  - A call that returns anything but W4A16_OK has launched nothing, except
 *    W4A16_ERR_CUDA from a failed launch (see w4a16_last_cuda_error()).
 *  - Group size G must be 32, 64 or 128, or equal to K (one scale per column);
 *    G = -1 is accepted as "equal to K". K must be a multiple of 8 (16-byte X
 *    rows) and N a multiple of 8 (16-byte Y rows). A shape whose tensor-core
 *    schedule would exceed 2^31 pipeline stages (about 2^31 * 16384 multiply-adds,
 *    far beyond device memory) is rejected with W4A16_ERR_INVALID_ARG.
 *  - The GEMM kernels are launched with programmatic dependent launch: a GEMM
 *    may start, and start streaming its packed weights, scales and zero-points,
 *    before the kernel enqueued just ahead of it on the stream has finished; it
 *    waits for that kernel before it reads x, bias or residual and before it
 *    writes y. So the kernel enqueued immediately before a GEMM on the same
 *    stream must not write that GEMM's packed weights, scales or zero-points.
 *    The repack calls (w4a16_pack, w4a16_pack_zeros, w4a16_sp_pack,
 *    w4a16_w8_pack) end with a kernel that writes nothing for this reason, so a
 *    GEMM may follow them directly. After writing packed buffers with a kernel
 *    of your own, enqueue another ordinary kernel (one launched without
 *    programmatic serialization) or synchronise before the GEMM.
 */
#ifndef W4A16_H
#define W4A16_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so the header needs no CUDA headers. */
struct CUstream_st;
typedef struct CUstream_st* w4a16_stream_t;

typedef enum {
    W4A16_OK = 0,
    W4A16_ERR_INVALID_ARG = 1,  /* a size, pointer, alignment or group size is invalid */
    W4A16_ERR_UNSUPPORTED = 2,  /* the device is not compute capability 10.3 (sm_103)  */
    W4A16_ERR_CUDA = 3,         /* a CUDA runtime call failed; code in w4a16_last_cuda_error() */
    W4A16_ERR_TIMEOUT = 4,      /* a kernel gave up waiting on one of its own pipeline barriers */
    W4A16_ERR_WORKSPACE = 5     /* the caller's workspace is smaller than w4a16_workspace_bytes() */
} w4a16_status;

/* Version of the packed layout written by w4a16_pack and read by the GEMM. Packed
 * buffers are a contract with this library: repack when the version changes. */
int w4a16_layout_version(void);

/* Static text for a status code. */
const char* w4a16_status_string(int status);

/* The cudaError_t of the last W4A16_ERR_CUDA returned on this host thread (0 if none). */
int w4a16_last_cuda_error(void);

/* Number of uint32 words of the packed weights: ceil(N/128) * KC * 1024, with
 * KC = ceil(K/64) rounded up to a multiple of 4 (K padded to a multiple of 256).
 * Returns 0 for invalid sizes. */
size_t w4a16_packed_words(int K, int N, int group_size);

/* Number of FP16 elements of the packed scales: ceil(N/128) * ceil(K/G) * 128.
 * Returns 0 for invalid sizes. */
size_t w4a16_scales_elems(int K, int N, int group_size);

/*
 * Repack codes and scales once, offline ("End-to-end flow": the layout is
 * computed once and exploited on every forward pass).
 *   codes          device, uint8 [K][N], values 0..15 (only the low nibble is read)
 *   scales         device, binary16 [ceil(K/G)][N] (or bfloat16 for w4a16_bf16_gemm:
 *                  the scales are copied as 16-bit patterns)
 *   packed         device out, uint32 [w4a16_packed_words(K, N, G)]
 *   scales_packed  device out, binary16 [w4a16_scales_elems(K, N, G)]
 * Packed layout (version 2): column tiles of 128 output features, reduction
 * chunks of 64. For tile nt, chunk kc, half j (32 values of k), feature n_in
 * and word w: word index (((nt*KC + kc)*2 + j)*128 + n_in)*4 + w with
 * KC = ceil(K/64) rounded up to a multiple of 4; the word holds
 * k0 = kc*64 + j*32 + w*8 .. k0+7 of column n = nt*128 + n_in, nibble i (bits 4i..4i+3) holding k = k0 + 2*(i%4) + i/4.
 * Positions outside K x N hold code 8 (weight 0). Scales: element
 * (nt*ceil(K/G) + g)*128 + n_in holds s[g][nt*128 + n_in] (0 outside N).
 */
w4a16_status w4a16_pack(const uint8_t* codes, const uint16_t* scales,
                        uint32_t* packed, uint16_t* scales_packed,
                        int K, int N, int group_size, w4a16_stream_t stream);

/*
 * Y = X x dequant(W), FP32 accumulation, FP16 output.
 *   x              device, binary16 [M][K]
 *   packed         device, output of w4a16_pack for (K, N, G)
 *   scales_packed  device, output of w4a16_pack for (K, N, G)
 *   y              device out, binary16 [M][N]; must not overlap the inputs
 * M = 0 is a no-op. Uses a per-device workspace that the library allocates on
 * the first call on each device (about 40 MB); make that first call outside
 * CUDA Graph capture. Calls on one device that run concurrently on different
 * streams share that workspace and must not overlap in time; use
 * w4a16_gemm_ws with separate workspaces for that. Repeated calls with equal
 * inputs give bit-identical outputs.
 */
w4a16_status w4a16_gemm(const uint16_t* x, const uint32_t* packed, const uint16_t* scales_packed,
                        uint16_t* y, int M, int N, int K, int group_size, w4a16_stream_t stream);

/* Bytes of caller workspace w4a16_gemm_ws needs for this shape, in any weight
 * format of this library (0 for invalid sizes). */
size_t w4a16_workspace_bytes(int M, int N, int K, int group_size);

/*
 * As w4a16_gemm, with a caller-owned device workspace of at least
 * w4a16_workspace_bytes(M, N, K, G) bytes, 256-byte aligned, ZEROED ONCE by the
 * caller before its first use; the kernels leave it ready for the next call.
 * This variant never allocates, so it can be captured into a CUDA Graph on
 * its first call. Returns W4A16_ERR_WORKSPACE if ws_bytes is too small.
 */
w4a16_status w4a16_gemm_ws(const uint16_t* x, const uint32_t* packed,
                           const uint16_t* scales_packed, uint16_t* y,
                           int M, int N, int K, int group_size,
                           void* workspace, size_t ws_bytes, w4a16_stream_t stream);

/* Activation of w4a16_gemm_fused, applied after the bias add. */
typedef enum {
    W4A16_ACT_NONE = 0,
    W4A16_ACT_SILU = 1, /* z / (1 + e^-z) */
    W4A16_ACT_RELU = 2  /* max(z, 0) */
} w4a16_activation;

/*
 * Y = act(X x dequant(W) + bias) + residual: the GEMM with the operations that
 * follow it in a layer fused into its epilogue ("quant_marlin_kernel", "End-to-end
 * flow": the output tile flows straight into a bias add and an activation), so Y
 * is written once instead of being re-read by separate kernels. The bias add, the
 * activation and the residual add run in FP32 on the accumulator; the result is
 * rounded once to FP16.
 *   bias       device, binary16 [N], or NULL for none
 *   residual   device, binary16 [M][N] row-major, or NULL for none; it may be the
 *              same buffer as y (an in-place y += ...) but must not otherwise
 *              overlap y
 *   activation a w4a16_activation
 *   workspace  as for w4a16_gemm_ws (ws_bytes bytes, zeroed once), or NULL to use
 *              the library's own workspace as w4a16_gemm does
 * Every other argument, layout and error is that of w4a16_gemm / w4a16_gemm_ws.
 * Returns W4A16_ERR_INVALID_ARG for an unknown activation or an odd bias or
 * residual address.
 */
w4a16_status w4a16_gemm_fused(const uint16_t* x, const uint32_t* packed,
                              const uint16_t* scales_packed, uint16_t* y,
                              int M, int N, int K, int group_size,
                              const uint16_t* bias, const uint16_t* residual, int activation,
                              void* workspace, size_t ws_bytes, w4a16_stream_t stream);

/*
 * w4a16_gemm_fused on row-strided activations, outputs and residual: X row m
 * starts at x + m * ldx, Y row m at y + m * ldy, residual row m at residual +
 * m * ldr (elements). A layer can read the leading K columns of a wider output
 * (the first 4096 of a fused QKV projection, the first 11008 of a gate/up
 * projection) and write into a slice of a wider buffer without a copy; the pages
 * have no counterpart (their kernels read contiguous activations).
 *   ldx  >= K, a multiple of 8 (rows start on 16-byte boundaries)
 *   ldy  >= N;   ldr >= N when residual is given (ignored otherwise)
 * Every other argument, layout and error is that of w4a16_gemm_fused; the rows of
 * Y must not overlap X or the residual (other than residual == y, same stride).
 * Returns W4A16_ERR_INVALID_ARG for strides outside these bounds.
 */
w4a16_status w4a16_gemm_strided(const uint16_t* x, int ldx, const uint32_t* packed,
                                const uint16_t* scales_packed, uint16_t* y, int ldy,
                                int M, int N, int K, int group_size,
                                const uint16_t* bias, const uint16_t* residual, int ldr, int activation,
                                void* workspace, size_t ws_bytes, w4a16_stream_t stream);

/* Bytes of the packed zero-points: ceil(N/128) * ceil(K/G) * 64 (two 4-bit
 * zero-points a byte). Returns 0 for invalid sizes. */
size_t w4a16_zeros_bytes(int K, int N, int group_size);

/*
 * Repack per-group zero-points once, offline, into the tile order the
 * zero-point GEMM streams beside the scales.
 *   zeros         device, uint8 [ceil(K/G)][N], values 0..15 (only the low nibble is read)
 *   zeros_packed  device out, uint8 [w4a16_zeros_bytes(K, N, G)], 16-byte aligned
 * Layout: byte (nt*ceil(K/G) + g)*64 + b holds z[g][nt*128 + 2b] in bits 0..3 and
 * z[g][nt*128 + 2b + 1] in bits 4..7; columns past N hold 8.
 * The codes and scales are packed by w4a16_pack as for the symmetric format.
 */
w4a16_status w4a16_pack_zeros(const uint8_t* zeros, uint8_t* zeros_packed, int K, int N, int group_size,
                              w4a16_stream_t stream);

/*
 * Y = act(X x dequant(W) + bias) + residual with per-group zero-points:
 * dequant(W)[k][n] = (q[k][n] - z[k/G][n]) * s[k/G][n]. (1024 + q) - (1024 + z)
 * is formed exactly in FP16, so the dequantised weight is rounded once, at the
 * product with the scale, as in the symmetric format.
 *   zeros_packed   device, output of w4a16_pack_zeros for (K, N, G); must not be NULL
 * Every other argument (bias, residual and activation may be NULL / 0 for a plain
 * GEMM; workspace NULL for the library's own), layout and error is that of
 * w4a16_gemm_fused. Zero-points all equal to 8 give bit-identical results to
 * w4a16_gemm_fused.
 */
w4a16_status w4a16_gemm_zp(const uint16_t* x, const uint32_t* packed, const uint16_t* scales_packed,
                           const uint8_t* zeros_packed, uint16_t* y, int M, int N, int K, int group_size,
                           const uint16_t* bias, const uint16_t* residual, int activation,
                           void* workspace, size_t ws_bytes, w4a16_stream_t stream);

/* ---------------------------------------------------------------- BF16 activations
 * The 4-bit GEMM (zero-point 8, layout of w4a16_pack) with every 16-bit tensor in
 * bfloat16 instead of binary16: X, the scales, bias, residual and Y, passed as
 * bfloat16 bit patterns (uint16_t). Both tensor-core operands are BF16: the weights
 * are dequantised to BF16, (128 + q) - 136 = q - 8 exactly, then one rounding at
 * the product with the scale (BF16 keeps 8 significant bits, so each weight
 * carries up to 2^-8 relative error against 2^-11 in the FP16 form).
 * ("Low-Precision Quantization Kernels in Production" (llms.blog), introduction:
 * FP16 and BF16 are the 16-bit types the weights are quantised from and the
 * tensor cores run.)
 *   scales_packed  w4a16_pack's scales output for BF16 scales (the repack copies
 *                  16-bit patterns, so the same call serves both types)
 * Every other argument, layout and error is that of w4a16_gemm_fused.
 */
w4a16_status w4a16_bf16_gemm(const uint16_t* x, const uint32_t* packed, const uint16_t* scales_packed,
                             uint16_t* y, int M, int N, int K, int group_size,
                             const uint16_t* bias, const uint16_t* residual, int activation,
                             void* workspace, size_t ws_bytes, w4a16_stream_t stream);

/* ---------------------------------------------------------------- 2:4 sparse 4-bit codes
 * Sparse-MARLIN ("MARLIN: Mixed-Precision Auto-Regressive Parallel Inference on
 * Large Language Models" note, key results: INT4 weights with 2:4 sparsity): the
 * 4-bit GEMM (zero-point 8, FP16) on codes that are 2:4 sparse along k, i.e. at
 * most two codes other than 8 (weight 0) in every aligned group of four k of a
 * column. Only two codes per group are stored, with their 2-bit positions, and
 * the sparse tensor-core MMA skips the other two: half the MMAs and 3/4 of the
 * weight bytes of the dense format. The result is that of w4a16_gemm_fused on the
 * same codes (exactly the same products, in another order of summation). */

/* Bytes of the sparse packed weights: ceil(N/128) * (KC/2) * 6144, KC as for
 * w4a16_packed_words. Returns 0 for invalid sizes. */
size_t w4a16_sp_packed_bytes(int K, int N, int group_size);

/*
 * Repack 2:4 sparse codes and scales once, offline.
 *   codes          device, uint8 [K][N], values 0..15, at most two codes other than 8
 *                  in every aligned group of four k of a column
 *   scales         device, binary16 [ceil(K/G)][N]
 *   packed         device out, uint8 [w4a16_sp_packed_bytes(K, N, G)], 16-byte aligned
 *   scales_packed  device out, binary16 [w4a16_scales_elems(K, N, G)] (as w4a16_pack)
 *   violations     device, 8-byte aligned counter, or NULL: the kernel adds the number
 *                  of groups that hold more than two codes other than 8 (those keep
 *                  their first two, so their results differ from the dense GEMM)
 * Sparse layout (version 1): chunks of 128 values of k (KC/2 per column), 6144
 * bytes per (column tile nt, chunk sc) at (nt*(KC/2) + sc)*6144:
 *   4096 bytes of stored codes: word ((b*128 + n_in)*4 + wd) holds stored values
 *     j0 = b*32 + wd*8 .. j0+7 of column nt*128 + n_in, nibble i holding stored
 *     value j0 + 2*(i%4) + i/4; stored value j is the code at k = 128*sc + 4*(j/2) +
 *     (position j%2 of group j/2);
 *   2048 bytes of position words, in the order the sparse MMA reads them from
 *     tensor memory: word (L*4 + mm), nibble u describes group t = 4*((L%16)/8) +
 *     u%4 of k = 128*sc + 32*mm + 4t .. +3 of column nt*128 + 16*(L/16) + 8*(u/4) +
 *     L%8: bits 0..1 the position (0..3) of the group's first stored code, bits
 *     2..3 that of its second (first < second).
 * A group stores the positions of its codes other than 8 in increasing order,
 * filled up to two with the smallest free positions (code 8). Padding (k >= K,
 * n >= N): code 8 at positions 0 and 1.
 */
w4a16_status w4a16_sp_pack(const uint8_t* codes, const uint16_t* scales, uint8_t* packed,
                           uint16_t* scales_packed, int K, int N, int group_size,
                           unsigned long long* violations, w4a16_stream_t stream);

/*
 * Y = act(X x dequant(W) + bias) + residual for 2:4 sparse codes packed by
 * w4a16_sp_pack. Arguments, epilogue and workspace as for w4a16_gemm_fused.
 */
w4a16_status w4a16_sp_gemm(const uint16_t* x, const uint8_t* packed, const uint16_t* scales_packed,
                           uint16_t* y, int M, int N, int K, int group_size,
                           const uint16_t* bias, const uint16_t* residual, int activation,
                           void* workspace, size_t ws_bytes, w4a16_stream_t stream);

/* ---------------------------------------------------------------- W8A16: 8-bit codes
 * The same GEMM for 8-bit weights: dequant(Wq)[k][n] = (q[k][n] - 128) * s[k/G][n],
 * q in 0..255, one FP16 scale per group ("Low-Precision Quantization Kernels in
 * Production" (llms.blog), section 1: the Marlin family serves 8-bit checkpoints
 * as well as 4-bit ones; 128 is the symmetric zero-point of unsigned 8-bit codes,
 * the pages print none). */

/* Bytes of the 8-bit packed codes: ceil(N/128) * KC * 8192, KC as for
 * w4a16_packed_words. Returns 0 for invalid sizes. */
size_t w4a16_w8_packed_bytes(int K, int N, int group_size);

/*
 * Repack 8-bit codes and scales once, offline.
 *   codes          device, uint8 [K][N], values 0..255
 *   scales         device, binary16 [ceil(K/G)][N]
 *   packed         device out, uint8 [w4a16_w8_packed_bytes(K, N, G)], 16-byte aligned
 *   scales_packed  device out, binary16 [w4a16_scales_elems(K, N, G)] (as w4a16_pack)
 * Packed layout (8-bit, version 1): column tiles of 128 output features, chunks of
 * 64 values of k, each in four quarters of 16. Byte
 * (((nt*KC + kc)*4 + j4)*128 + n_in)*16 + b belongs to word b/4, which holds
 * k0 = kc*64 + j4*16 + 4*(b/4) .. k0+3 of column nt*128 + n_in; bytes 0, 1, 2, 3 of
 * the word hold k0, k0+2, k0+1, k0+3. Positions outside K x N hold 128 (weight 0).
 */
w4a16_status w4a16_w8_pack(const uint8_t* codes, const uint16_t* scales, uint8_t* packed,
                           uint16_t* scales_packed, int K, int N, int group_size,
                           w4a16_stream_t stream);

/*
 * Y = act(X x dequant(W) + bias) + residual for 8-bit codes. (1024 + q) - 1152 is
 * q - 128 exactly in FP16; the dequantised weight is rounded once, at the product
 * with the scale.
 *   packed         device, output of w4a16_w8_pack for (K, N, G)
 * bias, residual, activation and workspace as for w4a16_gemm_fused (NULL / 0 for a
 * plain GEMM); w4a16_workspace_bytes covers this format too.
 */
w4a16_status w4a16_w8_gemm(const uint16_t* x, const uint8_t* packed, const uint16_t* scales_packed,
                           uint16_t* y, int M, int N, int K, int group_size,
                           const uint16_t* bias, const uint16_t* residual, int activation,
                           void* workspace, size_t ws_bytes, w4a16_stream_t stream);

/*
 * Synchronises `stream`, then reads and clears the error word that the kernels
 * set when one of their bounded waits gave up (W4A16_ERR_TIMEOUT), for the
 * given workspace. NULL covers the library's own workspace of the current device,
 * the error word of the kernels that run without a workspace (the decode and the
 * CUDA-core kernel) and, once a w4a16_gemm_noalloc call has run on that device,
 * the fixed array that call uses. After a timeout the split-K counters of the workspace (or
 * array) are reset as well.
 */
w4a16_status w4a16_check_device_status(void* workspace, w4a16_stream_t stream);

/*
 * Self-test of failure detection (no counterpart in the pages): launches one warp
 * that waits, with the kernels' own bounded wait, on a barrier that nothing ever
 * completes. After limit_ns (1 .. 10^10) the wait gives up, sets the error word of
 * `workspace` (NULL = the library's own workspace of the current device) and the
 * kernel returns; w4a16_check_device_status then reports W4A16_ERR_TIMEOUT and
 * clears it. The context stays usable. Nothing faults, traps or hangs.
 */
w4a16_status w4a16_selftest_wait_timeout(void* workspace, long long limit_ns, w4a16_stream_t stream);

/*
 * Sets the limit of every bounded wait in the kernels launched after this call
 * (default 1 s, or W4A16_WAIT_LIMIT_NS read at the first call on a device), for
 * tests of failure detection; no counterpart in the pages. A wait that runs out
 * makes its CTA give up: it stops issuing, waits (with a fixed 1 s bound) for the
 * copies and MMAs it already issued, frees its tensor memory and returns, and the
 * error word reports W4A16_ERR_TIMEOUT (w4a16_check_device_status); the results of
 * that launch are not valid. limit_ns <= 0 changes nothing. Returns the previous
 * limit. Applies to every device and host thread of the process.
 */
long long w4a16_set_wait_limit_ns(long long limit_ns);

/* Which kernel the dispatcher picks for a shape of the 4-bit FP16 format
 * (w4a16_gemm, w4a16_gemm_ws, w4a16_gemm_fused) on the current device. It picks
 * path 3 by itself for up to eight rows of X when K is a multiple of 32, and for up to
 * sixteen on layers of at most 4096 x 4096 with N >= 16 x the SM count (where it
 * measured faster on GB300), path 2 otherwise; path 1 only when forced:
 *   *path = 1: the CUDA-core kernel for one to four rows of X ("Low-Precision
 *              Quantization Kernels in Production" (llms.blog), section 2: the
 *              activation vector held on chip, weights streamed, unpacked in
 *              registers, group-scaled and reduced across a warp; section 5: at
 *              batch 1 the matmul is a memory-bound GEMV). *tile_m = the rows of X
 *              it is built for (1, 2 or 4); *grid = CTAs, one per block of 16 or
 *              32 output columns, each over the whole of K (no workspace is used).
 *   *path = 2: the tensor-core kernel (dequantised weights in tensor memory,
 *              tcgen05 MMA); *tile_m = rows of X per tile; *grid = CTAs.
 *   *path = 3: the decode kernel for one to sixteen rows of X ("quant_marlin_kernel",
 *              "The architecture": register-level unpack feeding the tensor-core
 *              MMA from registers; here warp-level MMAs). *tile_m = the rows of X
 *              it is built for (8 or 16); *grid = CTAs, one per block of 16 to 128
 *              output columns, each over the whole of K (no workspace is used).
 * The other weight formats always run path 2. */
w4a16_status w4a16_plan(int M, int N, int K, int group_size, int* path, int* tile_m, int* grid);

/* Forces the dispatcher's choice for the 4-bit FP16 format, for tests and
 * ablations (no counterpart in the pages): 0 = automatic (the default), 1 = the
 * CUDA-core kernel for every shape it serves (M <= 4), 2 = the tensor-core kernel
 * for every M, 3 = the decode kernel for every shape it serves (M <= 16, K a
 * multiple of 32). Shapes a forced path does not serve run path 2. Applies to every
 * later call in the process, on every device and host thread. Returns the previous
 * setting, or -1 (nothing changed) for another value. */
int w4a16_force_path(int path);

/*
 * w4a16_gemm without any device allocation by the library or the caller. The
 * pages have no counterpart; this entry point exists for callers that may not
 * allocate GPU memory at all: plug-ins whose host framework owns every byte of
 * device memory, and latency-critical loops that cannot afford cudaMalloc's
 * implicit device-wide synchronisation.
 *   Arguments, layouts and results are those of w4a16_gemm; the caller still
 *   passes x, packed, scales_packed and y.
 *   The split-K scratch of the tensor-core kernel (error word, tile counters,
 *   FP32 partials) lives in one fixed device array of W4A16_NOALLOC_MAX_BYTES
 *   inside the library, held by every GPU that loads the library until the
 *   process exits. A shape whose scratch would exceed it returns
 *   W4A16_ERR_WORKSPACE with nothing launched (on a 152-SM GB300 this admits
 *   every shape with M <= 32; at larger M only shapes the dispatcher gives few
 *   split tiles, such as 4096x12288 at M = 64; 4096x4096 at M = 64 needs
 *   8 MiB + 4352 bytes and is rejected). Shapes the decode kernel takes
 *   (M <= 8, K a multiple of 32) use no scratch at all, only its error word.
 *   The first call on each device looks the array's device address up; make
 *   that first call before any stream capture.
 *   A call that uses the scratch enqueues a clear of its tile counters, then the
 *   GEMM; the error word is left for w4a16_check_device_status(NULL, ...), which
 *   reads and clears it. Arguments are checked before anything is enqueued: a
 *   refused call touches nothing. Every call on a device shares the one array:
 *   calls whose work overlaps on the GPU (different streams, no ordering between
 *   them) race and give wrong results; order them on one stream or with events.
 *   Allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 */
#define W4A16_NOALLOC_MAX_BYTES ((size_t)8 << 20)
w4a16_status w4a16_gemm_noalloc(const uint16_t* x, const uint32_t* packed,
                                const uint16_t* scales_packed, uint16_t* y,
                                int M, int N, int K, int group_size, w4a16_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_H */
