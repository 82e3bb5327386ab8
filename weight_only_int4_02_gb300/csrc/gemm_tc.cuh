// W4A16 matmul on tcgen05 tensor cores, one persistent CTA per SM.
//
// Y[M][N] = X[M][K] * W[K][N], W[k][n] = (q - 8) * s[k/G][n], FP32 accumulate, FP16 out.
//
// The MMA runs "swapped": D[n][m] = sum_k W^T[n][k] * X^T[k][m], so the weight
// tile is the 128-row A operand and X supplies the N operand (TM rows of X,
// 16..256). A lives in tensor memory: dequant warps unpack the INT4 codes with
// bit operations (magic-number FP16 construction) straight into TMEM columns,
// so dequantised weights never touch shared memory; B (X) is loaded by TMA into
// 128-byte-swizzled shared memory; D accumulates in TMEM.
//
// A pipeline stage covers KSUB sub-chunks of 64 reduction values (KSUB = 4 for
// the memory-bound tiles, 2 for the compute-bound ones), so every barrier wait,
// commit and copy issue is paid once per 16 (or 8) MMAs.
//
// Warp roles (32 * (7 + 4*KSUB) threads):
//   warps 0-3           epilogue: TMEM -> registers -> FP16 Y, or FP32 partials + fix-up
//   warps 4 .. 4+4K-1   dequant, two teams taking alternate stages; a team has
//                       KSUB/2 groups of four warps (one per TMEM lane quarter),
//                       group g unpacking sub-chunks 2g and 2g+1 of its stages
//   next warp           producer X: TMA of the X tiles (one 3-D TMA per stage)
//   next warp           producer W: bulk copies of the packed words and the scales
//   last warp           MMA issuer (one elected lane) and TMEM owner
//
// Work split: whole waves of tiles go to the CTAs whole, round-robin; the tiles past
// them (the split region; every tile when there are fewer tiles than CTAs) have their
// (tile, stage) iterations cut into one contiguous range per CTA ("stream-K"), which
// each CTA runs before its whole tiles. A tile whose stages span several CTAs is
// reduced in global memory: every contributor stores its FP32 partial, and the last
// one to arrive on the tile's counter sums all partials in contributor order, so the
// result does not depend on arrival order.
//
// Sources: "quant_marlin_kernel" (aicassindra.com), "The architecture: every
// piece explained" (packed INT4, group scales, register-level unpack, async
// loads overlapped with MMA, split-K with a global reduction) and "End-to-end
// flow"; "Low-Precision Quantization Kernels in Production" (llms.blog),
// section 1 (offline pre-permuted layout, multi-stage pipeline, K-reduction
// adjusted to keep all SMs busy) and section 3 (deterministic split-K
// reduction in global memory).
#pragma once
#include <cuda.h>
#include "ptx.cuh"

namespace w4a16 {

constexpr int kTileN = 128;        // weight rows (output features) per tile = TMEM lanes
constexpr int kChunkK = 64;        // reduction values per sub-chunk
constexpr int kChunkWords = 1024;  // packed words per (tile, sub-chunk): 128 * 64 / 8
constexpr int kChunkBytes = 4096;
constexpr int kKPad = 4;           // the packed layout pads K to a multiple of 4 sub-chunks

// Weight formats (a template parameter of the kernel): 4-bit codes with the
// zero-point 8; 4-bit codes with one zero-point per (group, column); 8-bit codes
// with the zero-point 128 (8 KB per (tile, sub-chunk), bytes of a word in the
// order k, k+2, k+1, k+3); 4-bit codes with BF16 activations, scales and output;
// 2:4 sparse 4-bit codes (sub-chunks of 128 k: 4 KB of stored codes then 2 KB of
// position words in tensor-memory lane order, fed to the sparse MMA).
constexpr int kFmtW4 = 0;
constexpr int kFmtW4Zp = 1;
constexpr int kFmtW8 = 2;
constexpr int kFmtW4Bf16 = 3;   // 4-bit codes, zero-point 8, BF16 X / scales / bias / residual / Y
constexpr int kFmtW4Sp = 4;     // 4-bit codes, zero-point 8, 2:4 sparse along k (two stored per four)

struct GemmParams {
    const uint32_t* packed; // packed codes (4-bit: 1024 words per (tile, sub-chunk); 8-bit: 2048)
    const __half* scales;   // tile-ordered scales [n_tiles][ng][128]
    const uint8_t* zeros;   // tile-ordered 4-bit zero-points [n_tiles][ng][64 bytes] (kFmtW4Zp only)
    __half* y;              // 16-bit output (FP16, or BF16 bits for kFmtW4Bf16)
    float* partials;        // [2 * grid][TM][128] FP32
    int* counters;          // [grid], zero between launches (index = the tile's first contributor)
    int* status;            // error word, bit 0 = a wait timed out
    int M, N, K, G, ng;
    int g_shift;            // log2(G) for G a power of two; 30 when there is one group
    int n_tiles, m_tiles;
    int KC;                 // 64-value sub-chunks per weight column in the packed layout
    int iters;              // stages per tile = KC / KSUB
    int sk_tiles;           // tiles of the split region (the first ones), the rest whole
    long long sk_iters;     // sk_tiles * iters: the split region's stages
    int grid;               // CTAs: one work unit each
    int x_3d;               // X tensor map is 3-D {64, M, K/64}: one TMA per stage
    int x_rows;             // rows of X each TMA box brings (<= TM, a multiple of 8); the
                            // MMA's B rows past them feed only output columns >= M
    long long wait_limit_ns;
    // Fused epilogue, applied to every FP32 result before its rounding to FP16:
    // y = act(v + bias[n]) + residual[m][n]. Null pointers and act 0 leave v as is.
    const __half* bias;      // [N] or null
    const __half* residual;  // [M][ldr] or null (may be y itself)
    int act;                 // 0 none, 1 SiLU, 2 ReLU
    int ldy, ldr;            // row strides (elements) of y and the residual: >= N
};

// The fused epilogue on the FP32 result v: act(v + b) + r, with b and r already
// loaded (0 when absent). SiLU(z) = z / (1 + e^-z) with the fast exponential and
// division (about 2^-21 relative error). Callers load every bias and
// residual value they need before their stores of Y: the compiler cannot tell
// that those stores do not alias the loads, and would otherwise wait out each
// load after each store.
__device__ __forceinline__ float epilogue_op(int act, float v, float b, float r)
{
    v += b;
    if (act == 1)
        v = __fdividef(v, 1.f + __expf(-v));   // e^-v overflowing to inf gives -0, the limit
    else if (act == 2)
        v = fmaxf(v, 0.f);
    return v + r;
}

// 16-bit tensor elements: FP16, or BF16 bit patterns in the same storage (BF).
template <bool BF>
__device__ __forceinline__ float ld16(const __half* base, size_t i)
{
    if (!base) return 0.f;
    if constexpr (BF)
        return __uint_as_float((uint32_t)__half_as_ushort(base[i]) << 16);
    else
        return __half2float(base[i]);
}

template <bool BF>
__device__ __forceinline__ __half st16(float v)
{
    if constexpr (BF)
        return __ushort_as_half(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
    else
        return __float2half_rn(v);
}

template <int TM, int KSUB, int FMT = kFmtW4>
struct TcCfg {
    static constexpr bool kSp = FMT == kFmtW4Sp;
    static constexpr int kSubK = kSp ? 2 * kChunkK : kChunkK;   // values of k per sub-chunk
    static constexpr int kStageK = KSUB * kSubK;
    static constexpr int kXBlocks = kStageK / kChunkK;      // 64-wide K blocks of X per stage
    static constexpr int kXBlock = TM * 128;              // one 64-wide K block of X (TM rows)
    static constexpr int kXBytes = kXBlocks * kXBlock;
    // packed bytes per (tile, sub-chunk): 4-bit codes 4 KB, 8-bit codes 8 KB, 2:4
    // sparse 4 KB of stored codes + 2 KB of position words
    static constexpr int kPkChunk = FMT == kFmtW8 ? 2 * kChunkBytes : kSp ? kChunkBytes + 2048 : kChunkBytes;
    static constexpr int kPkBytes = KSUB * kPkChunk;
    static constexpr int kScBytes = (kStageK / 32) * 256;   // G = 32 puts kStageK/32 groups in a stage
    static constexpr int kZpBytes = FMT == kFmtW4Zp ? (kStageK / 32) * 64 : 0;  // 4-bit zero-points of those groups
    // Two rings in shared memory: W (packed words + scales [+ zero-points]), freed
    // by the dequant warps once they hold their words, so the HBM stream never
    // waits on the MMA; and X, freed by the MMA's commit.
    static constexpr int kWStageBytes = kPkBytes + kScBytes + kZpBytes;
    // a multiple of the team count; 8-bit stages of 128-row tiles and up are 4 deep
    // (64 KB of codes in flight, as 8 stages of 4-bit codes) to leave room for X.
    // 256-row tiles keep two: a stage of X is 64 KB there and one X slot more (three
    // instead of two) is worth more than W stages ahead, since each W stage feeds
    // 1024 cycles of MMAs (measured: 7-13% faster at M = 512 .. 4096).
    static constexpr int kWStages = (FMT == kFmtW8 || kSp) ? (TM >= 128 ? 4 : 8)
                                    : TM == 256                  ? 2
                                    : (TM <= 32 || KSUB == 2)    ? 8
                                                                 : 6;
    static constexpr int kXFit = (220 * 1024 - kWStages * kWStageBytes) / kXBytes;
    static constexpr int kXStages = kXFit > 8 ? 8 : kXFit;
    // Dequant teams take stages in turn; a team is KSUB/2 groups of four warps.
    static constexpr int kTeams = 2;
    static constexpr int kDqWarps = kTeams * 2 * KSUB;
    static constexpr int kDqWarp0 = 4;
    static constexpr int kProdXWarp = kDqWarp0 + kDqWarps;
    static constexpr int kProdWWarp = kProdXWarp + 1;
    static constexpr int kMmaWarp = kProdWWarp + 1;
    static constexpr int kThreads = 32 * (kMmaWarp + 1);
    static constexpr int kDBufs = TM <= 128 ? 2 : 1;
    // sparse: one position column per MMA, each at an 8-column boundary (the alignment
    // the MMA's A operand uses; a tighter packing has not been measured)
    static constexpr int kMetaStride = 8;
    static constexpr int kMetaCols = kSp ? KSUB * 4 * kMetaStride : 0;
    static constexpr int kASlotCols = KSUB * 32 + kMetaCols;  // 16-bit A values, two per column
    static constexpr int kAFit = (512 - kDBufs * TM) / kASlotCols;
    static constexpr int kAStages = kAFit >= 4 ? 4 : 2;               // a multiple of the team count
    static constexpr int kACol = 0;
    static constexpr int kDCol = kAStages * kASlotCols;
    static constexpr int kTmemCols = 512;
    // shared memory layout, offsets from a 1024-aligned base
    static constexpr int kOffX = 0;
    static constexpr int kOffPk = kOffX + kXStages * kXBytes;
    static constexpr int kOffSc = kOffPk + kWStages * kPkBytes;
    static constexpr int kOffZp = kOffSc + kWStages * kScBytes;
    static constexpr int kOffBar = kOffZp + kWStages * kZpBytes;
    // barriers: wfull[SW], wempty[SW], xfull[SX], xempty[SX], afull[A], aempty[A],
    // dfull[2], dempty[2], teardown
    static constexpr int kNumBars = 2 * kWStages + 2 * kXStages + 2 * kAStages + 4 + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + alignment slack
    static_assert(kXBlock % 1024 == 0, "X blocks must stay 1024-byte aligned");
    static_assert(kWStages >= 2 && kXStages >= 2 && kAStages >= 2, "pipeline depth");
    static_assert(kWStages % kTeams == 0 && kAStages % kTeams == 0, "rings shared by dequant teams in turn");
    static_assert(KSUB % 2 == 0, "a dequant warp unpacks two sub-chunks");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
    static_assert(kDCol + kDBufs * TM <= 512, "tensor memory");
    static_assert((kKPad * kChunkK) % kStageK == 0, "stages must tile the padded K");
    static_assert(!kSp || KSUB == 2, "sparse stages are two 128-value sub-chunks");
};

// Work of CTA c: first its range [cta_begin(c), cta_begin(c + 1)) of the split
// region's stages (tiles 0 .. sk_tiles-1, tile-major), then the whole tiles
// sk_tiles + c, sk_tiles + c + grid, ... The split region is every tile when there
// are fewer tiles than CTAs (each tile cut into the same number of parts), and the
// tiles past the last whole wave otherwise, so that a CTA's split work comes first:
// its partial and the tile's fix-up run under the MMAs of its whole tiles, and the
// launch ends on a whole tile's direct store.

// First split-region iteration of CTA c.
__device__ __forceinline__ long long cta_begin(const GemmParams& p, int c)
{
    return (long long)c * p.sk_iters / p.grid;
}

// The CTA whose range holds split-region iteration i.
__device__ __forceinline__ int cta_of(const GemmParams& p, long long i)
{
    int c = (int)((i * p.grid) / p.sk_iters);
    while (c + 1 < p.grid && cta_begin(p, c + 1) <= i) ++c;
    while (c > 0 && cta_begin(p, c) > i) --c;
    return c;
}

// Partial slot of CTA c for split tile t: 2c if t holds the CTA's first iteration, else 2c + 1.
__device__ __forceinline__ int slot_of(const GemmParams& p, int c, int t)
{
    return cta_begin(p, c) >= (long long)t * p.iters ? 2 * c : 2 * c + 1;
}

// Group of reduction index k, clamped to the last group (padding past K holds code 8).
__device__ __forceinline__ int group_of(const GemmParams& p, int k)
{
    return min(k >> p.g_shift, p.ng - 1);
}

__device__ __forceinline__ __half2 u32_as_half2(uint32_t u) { return *reinterpret_cast<const __half2*>(&u); }

// (q - 128) * s for 8-bit codes as two FP16 pairs (k, k+1), (k+2, k+3) from one
// word holding k, k+2, k+1, k+3 in bytes 0..3: OR-ing bytes 0 and 2 (or 1 and 3)
// into the mantissas of 1024.0 gives 1024 + q exactly (the ulp at 1024 is 1).
__device__ __forceinline__ void dequant_word8(uint32_t w, __half2 s2, uint32_t* out)
{
    const uint32_t mask = 0x00FF00FFu, magic = 0x64006400u;
    const __half2 c1152 = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    const uint32_t a = and_or(w, mask, magic);        // bytes 0, 2 -> k, k+1
    const uint32_t b = and_or(w >> 8, mask, magic);   // bytes 1, 3 -> k+2, k+3
    __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), c1152);
    __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), c1152);
    ha = __hmul2(ha, s2);
    hb = __hmul2(hb, s2);
    out[0] = *reinterpret_cast<uint32_t*>(&ha);
    out[1] = *reinterpret_cast<uint32_t*>(&hb);
}

// (q - 8) * s in BF16 as four pairs (k, k+1) ... (k+6, k+7) from one packed word
// (nibble i holds k + 2*(i%4) + i/4). BF16 keeps 7 fraction bits, so each nibble
// pair is shifted down to bits 0..3 of its half and OR-ed into 128.0 (0x4300):
// 128 + q exactly; (128 + q) - 136 is q - 8 exactly. s2 holds the scale's BF16 bits twice.
__device__ __forceinline__ void dequant_word_bf16(uint32_t w, uint32_t s2, uint32_t* out)
{
    const uint32_t lo = 0x000F000Fu, magic = 0x43004300u;
    const __nv_bfloat162 c136 = __halves2bfloat162(__ushort_as_bfloat16(0x4308), __ushort_as_bfloat16(0x4308));
    const __nv_bfloat162 sc = *reinterpret_cast<const __nv_bfloat162*>(&s2);
    uint32_t u[4] = {and_or(w, lo, magic), and_or(w >> 4, lo, magic), and_or(w >> 8, lo, magic),
                     and_or(w >> 12, lo, magic)};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 h = __hmul2(__hsub2(*reinterpret_cast<const __nv_bfloat162*>(&u[i]), c136), sc);
        out[i] = *reinterpret_cast<uint32_t*>(&h);
    }
}

// Dequantisation constants for the zero-point z (0..15), duplicated in both halves:
// lo = 1024 + z (binary16 0x6400 | z) and hi = -(64 + z) (0xD400 | 16z; the ulp at
// 64 is 1/16). z = 8 gives 1032 and -72.
__device__ __forceinline__ __half2 zp_lo(uint32_t z) { return u32_as_half2((0x6400u | z) * 0x00010001u); }
__device__ __forceinline__ __half2 zp_hi(uint32_t z) { return u32_as_half2((0xD400u | (z << 4)) * 0x00010001u); }

// (q - z) * s as four FP16 pairs (k, k+1) ... (k+6, k+7) from one packed word whose
// nibble i holds k + 2*(i%4) + i/4: OR-ing a nibble into the mantissa of 1024.0
// gives 1024 + q (low nibble of a byte) or 1024 + 16q (high nibble), both exact;
// (1024 + q) - (1024 + z) and (1024 + 16q) / 16 - (64 + z) are q - z exactly, and
// the one rounding is that of the product with the scale.
__device__ __forceinline__ void dequant_word(uint32_t w, __half2 s2, __half2 c_lo, __half2 c_hi, uint32_t* out)
{
    const uint32_t lo = 0x000F000Fu, hi = 0x00F000F0u, magic = 0x64006400u;
    const __half2 c1_16 = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
    const uint32_t w8 = w >> 8;
    const uint32_t a = and_or(w, lo, magic);   // nibbles 0, 4 -> k+0, k+1
    const uint32_t b = and_or(w, hi, magic);   // nibbles 1, 5 -> k+2, k+3
    const uint32_t c = and_or(w8, lo, magic);  // nibbles 2, 6 -> k+4, k+5
    const uint32_t d = and_or(w8, hi, magic);  // nibbles 3, 7 -> k+6, k+7
    __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), c_lo);
    __half2 hb = __hfma2(*reinterpret_cast<const __half2*>(&b), c1_16, c_hi);
    __half2 hc = __hsub2(*reinterpret_cast<const __half2*>(&c), c_lo);
    __half2 hd = __hfma2(*reinterpret_cast<const __half2*>(&d), c1_16, c_hi);
    ha = __hmul2(ha, s2);
    hb = __hmul2(hb, s2);
    hc = __hmul2(hc, s2);
    hd = __hmul2(hd, s2);
    out[0] = *reinterpret_cast<uint32_t*>(&ha);
    out[1] = *reinterpret_cast<uint32_t*>(&hb);
    out[2] = *reinterpret_cast<uint32_t*>(&hc);
    out[3] = *reinterpret_cast<uint32_t*>(&hd);
}

// One segment of a CTA's range: tile t, stages [kb, ke).
struct Segment {
    int t, kb, ke;
};

__device__ __forceinline__ Segment segment_at(const GemmParams& p, long long i, long long it_end)
{
    Segment g;
    g.t = (int)(i / p.iters);
    g.kb = (int)(i - (long long)g.t * p.iters);
    g.ke = (int)min((long long)p.iters, g.kb + (it_end - i));
    return g;
}

// A CTA's work as one run of local iterations v = 0 .. v_end: its split range of
// sk_len iterations from b = cta_begin(c) first, then its whole tiles, iters each.
// (The host keeps every count of stages below 2^31.)
__device__ __forceinline__ int work_len(const GemmParams& p, int c, int sk_len)
{
    const int tiles = p.n_tiles * p.m_tiles;
    const int whole = c + p.sk_tiles < tiles ? (tiles - p.sk_tiles - c + p.grid - 1) / p.grid : 0;
    return sk_len + whole * p.iters;
}

// The segment holding local iteration v of CTA c.
__device__ __forceinline__ Segment work_segment(const GemmParams& p, int c, long long b, int sk_len, int v)
{
    if (v < sk_len) return segment_at(p, b + v, b + sk_len);
    Segment g;
    g.t = p.sk_tiles + c + ((v - sk_len) / p.iters) * p.grid;
    g.kb = 0;
    g.ke = p.iters;
    return g;
}

// Epilogue stores of Y. An epilogue lane holds one output feature n (its TMEM lane)
// and 16 consecutive rows m of X (a tcgen05.ld of 16 columns), while Y is row-major in
// m with n contiguous, so a store straight from the registers writes 2 bytes per lane
// and row: 16 narrow stores per chunk, which measured about 1000 cycles per chunk with
// the GPU's memory busy. The chunk is transposed across lanes with shuffles first, so
// each lane stores two 16-byte vectors. FP32 partials keep their direct 4-byte stores
// (a warp writes 128 contiguous bytes per row; the transpose measured slower there, and
// a feature-major partial layout gave wrong sums on 128-row stream-K tiles: section 9).

// 8 x 8 transpose of 32-bit elements within each group of eight lanes: on return,
// x[k] of lane 8g + j is the x[j] that lane 8g + k held.
__device__ __forceinline__ void transpose8_lanes(uint32_t (&x)[8], int lane)
{
#pragma unroll
    for (int b = 4; b >= 1; b >>= 1) {
        const bool up = (lane & b) != 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (k & b) continue;
            const uint32_t recv = __shfl_xor_sync(0xffffffffu, up ? x[k] : x[k | b], b);
            if (up) x[k] = recv;
            else x[k | b] = recv;
        }
    }
}

// Rows m0 .. m0+15 of Y for the warp's 32 features n0 .. n0+31 (lane = feature), from
// the lane's FP32 accumulators r[e] (row m0 + e). After the transpose lane 8g + j holds
// rows m0 + 2j and m0 + 2j + 1 of features n0 + 8g .. +7 and writes each as one 16-byte
// vector (vec: Y rows 16-byte aligned), else element by element inside M and N.
template <bool BF>
__device__ __forceinline__ void store_y_rows16(const GemmParams& p, const uint32_t (&r)[16], int m0, int n0,
                                               int lane, bool vec)
{
    uint32_t h[8];   // h[k]: rows 2k (low half) and 2k+1 (high half), 16-bit
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float a = __uint_as_float(r[2 * k]), b = __uint_as_float(r[2 * k + 1]);
        if constexpr (BF) {
            const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
            h[k] = *reinterpret_cast<const uint32_t*>(&v);
        } else {
            const __half2 v = __floats2half2_rn(a, b);
            h[k] = *reinterpret_cast<const uint32_t*>(&v);
        }
    }
    transpose8_lanes(h, lane);   // h[k]: rows 2j, 2j+1 of feature 8g + k
    const int g = lane >> 3, j = lane & 7;
    const int n = n0 + 8 * g;
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
        const int m = m0 + 2 * j + hi;
        if (m >= p.M) continue;
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) o[q] = __byte_perm(h[2 * q], h[2 * q + 1], hi ? 0x7632u : 0x5410u);
        __half* dst = p.y + (size_t)m * p.ldy + n;
        if (vec && n + 8 <= p.N) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (n + e < p.N) dst[e] = __ushort_as_half((unsigned short)(o[e >> 1] >> (16 * (e & 1))));
        }
    }
}

// Rows m0 .. m0+15 of the residual for the warp's 32 features in the epilogue's layout
// (lane = feature, rv[e] = row m0 + e): lane 8g + j reads rows m0 + 2j and m0 + 2j + 1
// of features n0 + 8g .. +7 as two 16-byte vectors (vec: residual rows 16-byte
// aligned), else element by element, and the 8 x 8 transpose hands each lane its own
// feature's sixteen rows. Zero outside M and N or without a residual.
template <bool BF>
__device__ __forceinline__ void load_residual_rows16(const GemmParams& p, int m0, int n0, int lane, bool vec,
                                                     float (&rv)[16])
{
    const int g = lane >> 3, j = lane & 7;
    const int n = n0 + 8 * g;
    uint32_t w[2][4];
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
        const int m = m0 + 2 * j + hi;
        const __half* src = p.residual + (size_t)m * p.ldr + n;
        if (m < p.M && vec && n + 8 <= p.N) {
            const uint4 u = *reinterpret_cast<const uint4*>(src);
            w[hi][0] = u.x; w[hi][1] = u.y; w[hi][2] = u.z; w[hi][3] = u.w;
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t v = 0;
                if (m < p.M && n + 2 * q < p.N) v = __half_as_ushort(src[2 * q]);
                if (m < p.M && n + 2 * q + 1 < p.N) v |= (uint32_t)__half_as_ushort(src[2 * q + 1]) << 16;
                w[hi][q] = v;
            }
        }
    }
    uint32_t h[8];   // h[k]: rows 2j (low half) and 2j+1 (high half) of feature 8g + k
#pragma unroll
    for (int k = 0; k < 8; ++k) h[k] = __byte_perm(w[0][k >> 1], w[1][k >> 1], (k & 1) ? 0x7632u : 0x5410u);
    transpose8_lanes(h, lane);   // h[k]: rows 2k, 2k+1 of the lane's own feature
#pragma unroll
    for (int k = 0; k < 8; ++k) {
#pragma unroll
        for (int hi = 0; hi < 2; ++hi) {
            const uint32_t b16 = (h[k] >> (16 * hi)) & 0xffffu;
            if constexpr (BF)
                rv[2 * k + hi] = __uint_as_float(b16 << 16);
            else
                rv[2 * k + hi] = __half2float(__ushort_as_half((unsigned short)b16));
        }
    }
}

// Split-K fix-up of a tile by its last contributor: Y = the sum of every
// contributor's FP32 partial, added in contributor (CTA) order. Partials are
// [TM][128] per slot (row-major in m, the epilogue's lanes writing consecutive
// features). The nw participating warps (the four epilogue warps, or the whole CTA
// for its last tile) take (32-feature group, 16-row chunk) items in turn: a lane sums
// its feature's 16 rows over the contributors, NCP contributors' loads in flight at
// once (each load of a warp reads 128 contiguous bytes, one row of 32 features, from
// L2), and the warp writes the sums as the epilogue does (transposed across lanes,
// 16-byte stores). n_base is the tile's first feature.
template <int TM, int NCP, bool EPI, bool BF>
__device__ __forceinline__ void fix_tile(const GemmParams& p, int t, int c_lo, int c_hi, int valid, int m0, int n_base,
                                         int nw)
{
    const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
    const int chunks = (valid + 15) >> 4;
    const bool yvec = (p.ldy & 7) == 0;
    const bool rvec = ((reinterpret_cast<uintptr_t>(p.residual) | (uintptr_t)(p.ldr * 2)) & 15) == 0;
    for (int item = wi; item < 4 * chunks; item += nw) {
        const int fg = item & 3, c = item >> 2;
        const int n_in = fg * 32 + lane;
        float acc[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] = 0.f;
        for (int cc0 = c_lo; cc0 <= c_hi; cc0 += NCP) {
            float v[NCP][16];
#pragma unroll
            for (int u = 0; u < NCP; ++u) {
                const int cc = cc0 + u <= c_hi ? cc0 + u : c_hi;
                const float* a = p.partials + (size_t)slot_of(p, cc, t) * TM * kTileN + n_in + (size_t)c * 16 * kTileN;
#pragma unroll
                for (int e = 0; e < 16; ++e) v[u][e] = cc0 + u <= c_hi ? __ldcg(a + e * kTileN) : 0.f;
            }
#pragma unroll
            for (int u = 0; u < NCP; ++u) {
                if (cc0 + u > c_hi) break;
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[e] += v[u][e];
            }
        }
        uint32_t r[16];
        if constexpr (EPI) {
            const int n = n_base + n_in;
            const float bias_n = n < p.N ? ld16<BF>(p.bias, n) : 0.f;
            float rv[16];
            if (p.residual) {
                load_residual_rows16<BF>(p, m0 + c * 16, n_base + fg * 32, lane, rvec, rv);
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) rv[e] = 0.f;
            }
#pragma unroll
            for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(epilogue_op(p.act, acc[e], bias_n, rv[e]));
        } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(acc[e]);
        }
        store_y_rows16<BF>(p, r, m0 + c * 16, n_base + fg * 32, lane, yvec);
    }
}

// EPI: the instantiation with the fused epilogue (bias, activation, residual);
// the plain one carries none of its code.
template <int TM, int KSUB, bool EPI, int FMT>
__global__ void __launch_bounds__(TcCfg<TM, KSUB, FMT>::kThreads, 1)
    w4a16_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const GemmParams p)
{
    static_assert(FMT != kFmtW8 || KSUB == 2, "8-bit codes run 128-value stages (16 KB of codes)");
    constexpr bool ZP = FMT == kFmtW4Zp;
    constexpr bool BF = FMT == kFmtW4Bf16;
    using C = TcCfg<TM, KSUB, FMT>;
    constexpr int SW = C::kWStages;
    constexpr int SX = C::kXStages;
    constexpr int A = C::kAStages;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte-swizzled X tiles.
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
    const uint32_t sbase = smem_addr(smem);

    const uint32_t bar0 = sbase + C::kOffBar;
    auto wfull_bar = [&](int s) { return bar0 + 8u * s; };
    auto wempty_bar = [&](int s) { return bar0 + 8u * (SW + s); };
    auto xfull_bar = [&](int s) { return bar0 + 8u * (2 * SW + s); };
    auto xempty_bar = [&](int s) { return bar0 + 8u * (2 * SW + SX + s); };
    constexpr int kB1 = 2 * SW + 2 * SX;
    auto afull_bar = [&](int a) { return bar0 + 8u * (kB1 + a); };
    auto aempty_bar = [&](int a) { return bar0 + 8u * (kB1 + A + a); };
    auto dfull_bar = [&](int d) { return bar0 + 8u * (kB1 + 2 * A + d); };
    auto dempty_bar = [&](int d) { return bar0 + 8u * (kB1 + 2 * A + 2 + d); };
    const uint32_t teardown_bar = bar0 + 8u * (kB1 + 2 * A + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 16);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const WaitCtl ctl{abort_flag, p.status, p.wait_limit_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < SW; ++s) {
            mbar_init(wfull_bar(s), 1);
            mbar_init(wempty_bar(s), 2 * KSUB);      // the stage's dequant team (2*KSUB warps), once it holds its words
        }
        for (int s = 0; s < SX; ++s) {
            mbar_init(xfull_bar(s), 1);
            mbar_init(xempty_bar(s), 1);             // the MMA commit
        }
        for (int a = 0; a < A; ++a) {
            mbar_init(afull_bar(a), 2 * KSUB);       // the stage's dequant team
            mbar_init(aempty_bar(a), 1);
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(dfull_bar(d), 1);
            mbar_init(dempty_bar(d), 4);
        }
        mbar_init(teardown_bar, 1);
        *abort_flag = 0;
        reinterpret_cast<int*>(smem + C::kOffMisc + 24)[0] = 0;   // no deferred fix-up yet
        fence_mbar_init();
    }
    if (warp == C::kProdXWarp && lane == 0) prefetch_tmap(&tmap_x);
    if (warp == C::kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (threadIdx.x == 0) launch_dependents();

    const int cta = blockIdx.x;
    const long long it_begin = cta_begin(p, cta);
    const int sk_len = (int)(cta_begin(p, cta + 1) - it_begin);
    const int v_end = work_len(p, cta, sk_len);

    // Every role walks the same stage sequence seq = 0, 1, ... over the CTA's
    // range; stage seq uses slot seq % S of the shared ring and slot seq % A of
    // the TMEM A ring. Each role visits every seq in order, so no waiter can be
    // a whole phase ahead of a barrier (parity waits cannot tell p from p + 2).
    if (warp == C::kProdXWarp || warp == C::kProdWWarp) {
        // ------------------------------------------------------------ producers
        // W streams packed words and scales, which no earlier kernel writes, so it
        // starts at once; X may be the previous kernel's output, so the X producer
        // first waits for that kernel to complete.
        const bool is_x = warp == C::kProdXWarp;
        if (is_x) wait_prior_grid();
        const int S = is_x ? SX : SW;
        uint32_t seq = 0;
        bool ok = true;
        for (int v = 0; ok && v < v_end;) {
            const Segment g = work_segment(p, cta, it_begin, sk_len, v);
            const int nt = g.t / p.m_tiles, mt = g.t - nt * p.m_tiles;
            for (int kc = g.kb; kc < g.ke; ++kc, ++seq) {
                const int s = (int)(seq % S);
                const uint32_t empty = is_x ? xempty_bar(s) : wempty_bar(s);
                if (!wait_warp(empty, ((seq / S) & 1) ^ 1, ctl)) { ok = false; break; }
                if (lane == 0) {
                    const int k0 = kc * C::kStageK;
                    if (is_x) {
                        mbar_arrive_expect_tx(xfull_bar(s), (uint32_t)(C::kXBlocks * p.x_rows * 128));
                        if (p.x_3d) {
                            tma_load_3d(sbase + C::kOffX + s * C::kXBytes, &tmap_x, xfull_bar(s), 0, mt * TM,
                                        kc * C::kXBlocks);
                        } else {
#pragma unroll
                            for (int j = 0; j < C::kXBlocks; ++j)
                                tma_load_2d(sbase + C::kOffX + s * C::kXBytes + j * p.x_rows * 128, &tmap_x,
                                            xfull_bar(s), k0 + j * kChunkK, mt * TM);
                        }
                    } else {
                        const int g0 = group_of(p, k0);
                        const int g1 = group_of(p, k0 + C::kStageK - 1);
                        const uint32_t sc_bytes = (uint32_t)(g1 - g0 + 1) * 256u;
                        const uint32_t zp_bytes = ZP ? (uint32_t)(g1 - g0 + 1) * 64u : 0u;
                        mbar_arrive_expect_tx(wfull_bar(s), C::kPkBytes + sc_bytes + zp_bytes);
                        bulk_load(sbase + C::kOffPk + s * C::kPkBytes,
                                  p.packed + ((size_t)nt * p.KC + (size_t)kc * KSUB) * (C::kPkChunk / 4),
                                  C::kPkBytes, wfull_bar(s));
                        bulk_load(sbase + C::kOffSc + s * C::kScBytes, p.scales + ((size_t)nt * p.ng + g0) * kTileN,
                                  sc_bytes, wfull_bar(s));
                        if constexpr (ZP)
                            bulk_load(sbase + C::kOffZp + s * C::kZpBytes, p.zeros + ((size_t)nt * p.ng + g0) * 64,
                                      zp_bytes, wfull_bar(s));
                    }
                }
                __syncwarp();
            }
            v += g.ke - g.kb;
        }
        // Wind down: let the last copies land before the CTA can exit.
        if (lane == 0) {
            const uint32_t inflight = seq < (uint32_t)S ? seq : (uint32_t)S;
            for (uint32_t k = 1; k <= inflight; ++k) {
                const uint32_t q = seq - k;
                wait_drain(is_x ? xfull_bar((int)(q % S)) : wfull_bar((int)(q % S)), (q / S) & 1, 1000000000LL);
            }
        }
    } else if (warp == C::kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        constexpr uint32_t idesc =
            (BF ? idesc_bf16_f32(128, TM) : idesc_f16_f32(128, TM)) | (C::kSp ? kIdescSparse : 0u);
        uint32_t seq = 0;
        int d = 0;
        uint32_t dph = 0;
        bool ok = true;
        for (int v = 0; ok && v < v_end;) {
            const Segment g = work_segment(p, cta, it_begin, sk_len, v);
            if (!wait_warp(dempty_bar(d), dph ^ 1, ctl)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + C::kDCol + d * TM;
            for (int kc = g.kb; kc < g.ke; ++kc, ++seq) {
                const int s = (int)(seq % SX);
                const int a = (int)(seq % A);
                if (!wait_warp(xfull_bar(s), (seq / SX) & 1, ctl) || !wait_warp(afull_bar(a), (seq / A) & 1, ctl)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    const uint64_t b0 = smem_desc_k_sw128(sbase + C::kOffX + s * C::kXBytes);
                    const uint32_t a0 = tmem + C::kACol + a * C::kASlotCols;
                    // The descriptor's start address counts 16-byte units: +2 per 16 K values
                    // inside a 128-byte row, +x_rows*128/16 per 64-wide K block (blocks of
                    // x_rows rows sit back to back, each 1024-byte aligned).
                    if constexpr (C::kSp) {
                        // sub-chunk j: 4 sparse MMAs of 32 values of k, each reading 8 A columns
                        // (16 stored values), one position column, and half an X block (+4 per 32 k)
#pragma unroll
                        for (int j = 0; j < KSUB; ++j) {
#pragma unroll
                            for (int mm = 0; mm < 4; ++mm) {
                                const uint64_t bd = b0 + (uint64_t)((2 * j + mm / 2) * p.x_rows * 8 + (mm % 2) * 4);
                                mma_f16_sp_ts(d_tmem, a0 + j * 32 + mm * 8, bd,
                                              a0 + KSUB * 32 + (j * 4 + mm) * C::kMetaStride, idesc,
                                              (kc > g.kb || j > 0 || mm > 0) ? 1u : 0u);
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < KSUB; ++j) {
#pragma unroll
                            for (int kk = 0; kk < kChunkK / 16; ++kk) {
                                const uint64_t bd = b0 + (uint64_t)(j * p.x_rows * 8 + kk * 2);
                                mma_f16_ts(d_tmem, a0 + j * 32 + kk * 8, bd, idesc,
                                           (kc > g.kb || j > 0 || kk > 0) ? 1u : 0u);
                            }
                        }
                    }
                    mma_commit(xempty_bar(s));
                    mma_commit(aempty_bar(a));
                }
                __syncwarp();
            }
            if (!ok) break;
            if (elect_one()) mma_commit(dfull_bar(d));
            __syncwarp();
            if (++d == C::kDBufs) { d = 0; dph ^= 1; }
            v += g.ke - g.kb;
        }
        // Wind down: every MMA issued so far completes before TMEM is freed.
        if (lane == 0) {
            mma_commit(teardown_bar);
            wait_drain(teardown_bar, 0, 1000000000LL);
        }
    } else if (warp >= C::kDqWarp0) {
        // ------------------------------------------------------------ dequant
        // Teams take stages in turn, so one team's waits overlap the others'
        // arithmetic. Within a team, group gi unpacks sub-chunks 2gi and 2gi+1.
        // Ring depths are multiples of the team count: a ring slot's successive uses
        // all fall to one team, which visits its stages in order (no waiter is a
        // whole phase ahead).
        constexpr int kWarpsPerTeam = 2 * KSUB;
        const int dw = warp - C::kDqWarp0;
        const int team = dw / kWarpsPerTeam;
        const int gi = (dw % kWarpsPerTeam) >> 2;
        const int quarter = warp & 3;                // TMEM lanes 32*quarter .. +31
        const int n_in = quarter * 32 + lane;
        const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
        uint32_t seq = 0;
        bool ok = true;
        for (int v = 0; ok && v < v_end;) {
            const Segment g = work_segment(p, cta, it_begin, sk_len, v);
            for (int kc = g.kb; kc < g.ke; ++kc, ++seq) {
                if ((int)(seq % C::kTeams) != team) continue;
                const int s = (int)(seq % SW);
                const int a = (int)(seq % A);
                if (!wait_warp(wfull_bar(s), (seq / SW) & 1, ctl)) { ok = false; break; }
                const int gs = group_of(p, kc * C::kStageK);
                const __half* sc = reinterpret_cast<const __half*>(smem + C::kOffSc + s * C::kScBytes) + n_in;
                const uint8_t* zb = smem + C::kOffZp + s * C::kZpBytes + (n_in >> 1);   // ZP only
                const int zshift = 4 * (n_in & 1);
                // A thread's 16-byte blocks of a sub-chunk sit 2 KB apart: 2 for 4-bit
                // codes (32 values each; 32 stored values of 64 k when sparse), 4 for
                // 8-bit codes (16 values each). Sparse sub-chunks then hold the
                // thread's lane of position words (16 bytes per lane).
                constexpr int NB = FMT == kFmtW8 ? 4 : 2;
                constexpr int NS = C::kSubK / 32;   // scales per sub-chunk (one per 32 k; G >= 32)
                uint4 w[2][NB];
                uint4 meta[2];
                __half2 s2[2][NS];
                __half2 clo[2][2], chi[2][2];
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int j = 2 * gi + h;
                    const uint8_t* pk = smem + C::kOffPk + s * C::kPkBytes + j * C::kPkChunk + n_in * 16;
#pragma unroll
                    for (int b = 0; b < NB; ++b) w[h][b] = *reinterpret_cast<const uint4*>(pk + b * kTileN * 16);
                    if constexpr (C::kSp) meta[h] = *reinterpret_cast<const uint4*>(pk + kChunkBytes);
                    const int k0 = kc * C::kStageK + j * C::kSubK;
#pragma unroll
                    for (int q = 0; q < NS; ++q) {
                        const __half sq = sc[(group_of(p, k0 + 32 * q) - gs) * kTileN];
                        s2[h][q] = __halves2half2(sq, sq);
                    }
                    if constexpr (ZP) {
                        const uint32_t z_lo = (zb[(group_of(p, k0) - gs) * 64] >> zshift) & 0xFu;
                        const uint32_t z_hi = (zb[(group_of(p, k0 + 32) - gs) * 64] >> zshift) & 0xFu;
                        clo[h][0] = zp_lo(z_lo);
                        chi[h][0] = zp_hi(z_lo);
                        clo[h][1] = zp_lo(z_hi);
                        chi[h][1] = zp_hi(z_hi);
                    } else {
                        clo[h][0] = clo[h][1] = zp_lo(8);
                        chi[h][0] = chi[h][1] = zp_hi(8);
                    }
                }
                fence_proxy_async_smem();   // the loads above precede the slot's next bulk copy
                __syncwarp();
                if (lane == 0) mbar_arrive(wempty_bar(s));   // words, scales and zero-points are in registers
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t v[32];   // FP16 pairs (k, k+1) of the sub-chunk's 64 values
                    if constexpr (BF) {
#pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            const uint32_t sb = *reinterpret_cast<const uint32_t*>(&s2[h][b]);
                            dequant_word_bf16(w[h][b].x, sb, v + 16 * b + 0);
                            dequant_word_bf16(w[h][b].y, sb, v + 16 * b + 4);
                            dequant_word_bf16(w[h][b].z, sb, v + 16 * b + 8);
                            dequant_word_bf16(w[h][b].w, sb, v + 16 * b + 12);
                        }
                    } else if constexpr (C::kSp) {
                        // stored values: word (b, wd) holds 8 of groups covering k b*64 + wd*16 .. +15
#pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            dequant_word(w[h][b].x, s2[h][2 * b], clo[h][0], chi[h][0], v + 16 * b + 0);
                            dequant_word(w[h][b].y, s2[h][2 * b], clo[h][0], chi[h][0], v + 16 * b + 4);
                            dequant_word(w[h][b].z, s2[h][2 * b + 1], clo[h][0], chi[h][0], v + 16 * b + 8);
                            dequant_word(w[h][b].w, s2[h][2 * b + 1], clo[h][0], chi[h][0], v + 16 * b + 12);
                        }
                    } else if constexpr (FMT == kFmtW8) {
#pragma unroll
                        for (int b = 0; b < 4; ++b) {
                            dequant_word8(w[h][b].x, s2[h][b >> 1], v + 8 * b + 0);
                            dequant_word8(w[h][b].y, s2[h][b >> 1], v + 8 * b + 2);
                            dequant_word8(w[h][b].z, s2[h][b >> 1], v + 8 * b + 4);
                            dequant_word8(w[h][b].w, s2[h][b >> 1], v + 8 * b + 6);
                        }
                    } else {
                        dequant_word(w[h][0].x, s2[h][0], clo[h][0], chi[h][0], v + 0);
                        dequant_word(w[h][0].y, s2[h][0], clo[h][0], chi[h][0], v + 4);
                        dequant_word(w[h][0].z, s2[h][0], clo[h][0], chi[h][0], v + 8);
                        dequant_word(w[h][0].w, s2[h][0], clo[h][0], chi[h][0], v + 12);
                        dequant_word(w[h][1].x, s2[h][1], clo[h][1], chi[h][1], v + 16);
                        dequant_word(w[h][1].y, s2[h][1], clo[h][1], chi[h][1], v + 20);
                        dequant_word(w[h][1].z, s2[h][1], clo[h][1], chi[h][1], v + 24);
                        dequant_word(w[h][1].w, s2[h][1], clo[h][1], chi[h][1], v + 28);
                    }
                    if (h == 0) {
                        // the A slot is free once the MMAs that read it two stages ago completed
                        if (!wait_warp(aempty_bar(a), ((seq / A) & 1) ^ 1, ctl)) { ok = false; break; }
                        tc_fence_after();
                    }
                    tmem_st32(tmem + lane_base + C::kACol + a * C::kASlotCols + (2 * gi + h) * 32, v);
                    if constexpr (C::kSp) {
                        const uint32_t mcol = tmem + lane_base + C::kACol + a * C::kASlotCols + KSUB * 32 +
                                              (2 * gi + h) * 4 * C::kMetaStride;
                        tmem_st1(mcol + 0 * C::kMetaStride, meta[h].x);
                        tmem_st1(mcol + 1 * C::kMetaStride, meta[h].y);
                        tmem_st1(mcol + 2 * C::kMetaStride, meta[h].z);
                        tmem_st1(mcol + 3 * C::kMetaStride, meta[h].w);
                        tmem_wait_st();
                    }
                }
                if (!ok) break;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(afull_bar(a));
            }
            v += g.ke - g.kb;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int n_in = warp * 32 + lane;
        int d = 0;
        uint32_t dph = 0;
        for (int v = 0; v < v_end;) {
            const Segment g = work_segment(p, cta, it_begin, sk_len, v);
            const int t = g.t;
            const int nt = t / p.m_tiles, mt = t - nt * p.m_tiles;
            const int n = nt * kTileN + n_in;
            const int m0 = mt * TM;
            const int valid = min(TM, p.M - m0);
            const int chunks = (valid + 15) >> 4;
            const bool split = (g.kb != 0 || g.ke != p.iters);
            // The bias of this row is fetched while the MMAs run.
            const float bias_n = (EPI && n < p.N) ? ld16<BF>(p.bias, n) : 0.f;
            // All four epilogue warps leave together: they share named barriers.
            const bool ok = wait_warp(dfull_bar(d), dph, ctl);
            if (named_bar_or(1, 128, !ok)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + ((uint32_t)(warp * 32) << 16) + C::kDCol + d * TM;
            float* part = p.partials + (size_t)slot_of(p, cta, t) * TM * kTileN + n_in;
            const bool yvec = (p.ldy & 7) == 0;   // Y rows 16-byte aligned (Y itself is)
            const bool rvec = ((reinterpret_cast<uintptr_t>(p.residual) | (uintptr_t)(p.ldr * 2)) & 15) == 0;
            for (int c = 0; c < chunks; ++c) {
                uint32_t r[16];
                tmem_ld16(d_tmem + c * 16, r);
                if (!split) {
                    if constexpr (EPI) {
                        float rv[16];
                        if (p.residual) {
                            load_residual_rows16<BF>(p, m0 + c * 16, n - lane, lane, rvec, rv);
                        } else {
#pragma unroll
                            for (int e = 0; e < 16; ++e) rv[e] = 0.f;
                        }
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            r[e] = __float_as_uint(epilogue_op(p.act, __uint_as_float(r[e]), bias_n, rv[e]));
                    }
                    store_y_rows16<BF>(p, r, m0 + c * 16, n - lane, lane, yvec);
                } else {
                    // the lane's 16 rows of the chunk, contiguous in its feature's row of the slot
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (c * 16 + e < valid) part[(size_t)(c * 16 + e) * kTileN] = __uint_as_float(r[e]);
                }
            }
            // The accumulator is free once its values are in global memory; the
            // fix-up reads every partial, this CTA's own included, back from L2.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty_bar(d));
            if (++d == C::kDBufs) { d = 0; dph ^= 1; }
            v += g.ke - g.kb;

            if (split) {
                // Deterministic split-K fix-up: the last contributor sums every
                // contributor's partial in CTA order.
                __threadfence();
                named_bar_sync(1, 128);
                const int c_lo = cta_of(p, (long long)t * p.iters);
                const int c_hi = cta_of(p, (long long)t * p.iters + p.iters - 1);
                if (threadIdx.x == 0) {
                    int* counter = p.counters + c_lo;
                    const int prev = atomicAdd(counter, 1);
                    const int last = (prev == c_hi - c_lo);
                    if (last) *counter = 0;
                    *last_flag = last;
                }
                named_bar_sync(1, 128);
                const int last = *last_flag;
                if (last && v >= v_end) {
                    // the CTA's final tile: every warp reduces it once all roles are done
                    if (threadIdx.x == 0) {
                        int* dfr = reinterpret_cast<int*>(smem + C::kOffMisc + 24);
                        dfr[0] = 1; dfr[1] = t; dfr[2] = c_lo; dfr[3] = c_hi;
                    }
                } else if (last) {
                    __threadfence();
                    fix_tile<TM, KSUB == 4 ? 2 : 4, EPI, BF>(p, t, c_lo, c_hi, valid, m0, n - n_in, 4);
                }
                named_bar_sync(1, 128);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    {
        // the split-K fix-up of the CTA's final tile, if it arrived last, by all warps
        const int* dfr = reinterpret_cast<const int*>(smem + C::kOffMisc + 24);
        if (dfr[0]) {
            __threadfence();
            const int t = dfr[1];
            const int nt = t / p.m_tiles, mt = t - nt * p.m_tiles;
            const int m0 = mt * TM;
            fix_tile<TM, KSUB == 4 ? 2 : 4, EPI, BF>(p, t, dfr[2], dfr[3], min(TM, p.M - m0), m0, nt * kTileN,
                                                     C::kThreads / 32);
        }
    }
    if (warp == C::kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int TM, int KSUB, bool EPI, int FMT>
cudaError_t launch_tc(const CUtensorMap& tmap, const GemmParams& p, cudaStream_t stream);

template <int TM, int KSUB, bool EPI, int FMT>
cudaError_t setup_tc();

}  // namespace w4a16
