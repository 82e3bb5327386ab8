// W4A16 matmul for one to sixteen rows of X: register-level unpack of the INT4
// codes into the operand registers of warp-level MMAs (no tensor memory, no
// split-K workspace).
//
// Y[m][n] = sum_g s[g][n] * sum_{k in g} X[m][k] * (q[k][n] - 8), FP32 accumulate, FP16 out.
//
// With a few rows of X the matmul streams the packed weights from HBM and uses
// each of them M times. On this GPU the tensor-memory MMA costs a fixed number of
// cycles per instruction below 64 columns of X, which caps the 4-bit stream of the
// tensor-core kernel under the HBM rate; a warp-level MMA
// (mma.sync.m16n8k16, FP16 x FP16 -> FP32) fed from registers has no such floor
// at this size, so this kernel spends its issue slots on the unpack alone: nine
// instructions per packed word of eight codes, and one MMA per 256 weights and
// eight rows of X.
//
// Operands. The MMA runs "swapped": A = 16 weight columns (output features) x 16
// values of k, B = 16 values of k x 8 rows of X, D[n][m] in FP32. The packed layout
// (version 2, the one the tensor-core kernel reads) keeps eight consecutive values
// of k of one column in a word, nibbles (0,4) (1,5) (2,6) (3,7) holding the pairs
// (k, k+1) ... (k+6, k+7). Lane (g, t) = (lane / 4, lane % 4) of a warp takes word t
// of a 32-value row for column g and for column g + 8 of a 16-column block; the
// magic-number unpack (OR a nibble pair into the mantissas of 1024.0, subtract
// 1032; the high nibbles through 1024 + 16q) turns each word into four exact FP16
// pairs of (q - 8). They form the A registers of two MMAs when the MMA's k-slots
// (2t, 2t+1) and (2t+8, 2t+9) are taken to mean the values 8t + (0,1) and 8t + (2,3)
// of the row (first MMA) and 8t + (4,5), 8t + (6,7) (second MMA). The B registers
// follow the same meaning of the k-slots: lane (g, t) supplies X[g][8t .. 8t+7] of
// the row, one 16-byte load. The sum over k does not depend on which slot carries
// which k, so D is the exact sum of (q - 8) * X over the row's 32 values, for 16
// columns and 8 rows of X (a second pair of MMAs takes rows 8..15).
//
// Group scales are applied in FP32 to the MMA sums: each warp sums the values of k
// of one group it takes from a stage (128 when G >= 128, else G) in accumulators
// whose first MMA starts from zero, and adds them, times the group's scale, to its
// running sums. Products of (q - 8) and X are exact in the MMA; the scale multiplies
// once per group.
//
// Work split: the output columns are cut into blocks of CB (16, 32, 48, 64, 80 or
// 128); one CTA takes one block over the whole of K, so no partial sum leaves the
// CTA. A stage is 16 rows of 32 values of k (512 values); two teams of four consumer
// warps take the stages in turn, warp w of a team rows 4w .. 4w+3 (128 values of k)
// for all CB columns; with 128 columns both teams take every stage, each 64 of the
// columns. At the end the warps' sums are added in warp order through shared memory
// (bit-identical results from run to run).
//
// Staging: one producer warp streams the stage's packed words (2-D TMA boxes of 16
// rows x up to 64 columns, each inside one 128-column tile) and group scales into a
// ring of 24 to 80 KB of words (by block width); it needs nothing from the previous
// kernel, so the ring fills while that kernel finishes (programmatic dependent
// launch). With an odd number of slots a team first waits for the other team to
// consume a slot's earlier stage. A second producer waits for the previous kernel, then brings
// the stage's X with one 3-D TMA as [16 rows][mr rows of X][32 values]: 64 bytes per
// row of X, so the eight rows a quarter-warp reads sit in different banks.
// A CTA holds under half of an SM (about 100 KB of shared memory, 320 threads), so
// two run side by side and the next launch's CTAs start as soon as a slot frees.
//
// Every wait is bounded: a wait that runs out sets the CTA's abort flag and the
// launch's error word; the consumers skip the remaining rows, the producers stop
// issuing, wait (bounded) for their copies in flight, and the CTA returns.
//
// Sources: "quant_marlin_kernel" (aicassindra.com), "The architecture: every
// piece explained" (packed INT4, group scales, register-level unpack with bit
// operations, FP16 activations in and out, tensor-core MMA fed from registers) and
// "End-to-end flow"; "Low-Precision Quantization Kernels in Production"
// (llms.blog), section 1 (pre-permuted layout so one load lands in MMA operand
// order, multi-stage asynchronous pipeline) and section 5 ("Decoding Roofline
// Dynamics": at small batch the matmul is bound by the weight stream).
#include <cuda.h>
#include <cuda_runtime.h>

#include "decode.cuh"
#include "gemm_tc.cuh"

namespace w4a16 {

namespace {

constexpr int kConsumers = 8;
constexpr int kProdW = kConsumers;
constexpr int kProdX = kConsumers + 1;
static_assert(kDecThreads == 32 * (kConsumers + 2), "warp roles");
static_assert(kDecStageRows == 2 * kConsumers, "two rows of a stage per consumer warp");

// Shared memory: [ring][CB / box][16][box][16 bytes] packed words (one TMA box of
// `box` columns each), [ring][16][CB] scales (or [CB / 16][16][16] with 16-column
// boxes), [ring][16][x_rows][64 bytes] X, then the barriers. The ring depth and X's
// rows are launch parameters (offsets computed at run time). With 128-column blocks
// the two consumer teams split the columns (64 each) and both take every stage; with
// 16 to 80 they take the stages in turn over all columns. Blocks of 48 and 80 columns
// can straddle two 128-column tiles of the packed layout: their words and scales come
// in boxes of 16 columns, each within one tile.
template <int MR, int CB>
struct DecCfg {
    static constexpr bool kColTeams = CB == 128;
    static constexpr bool kNarrowBoxes = CB == 48 || CB == 80;
    static constexpr int kWarpCols = kColTeams ? 64 : CB;     // output columns of one consumer warp
    static constexpr int kBoxCols = kNarrowBoxes ? 16 : CB > 64 ? 64 : CB;   // columns of one weight TMA box
    static constexpr int kBoxBytes = kDecStageRows * kBoxCols * 16;
    static constexpr int kSBoxHalves = kDecStageRows * 16;   // one 16-column box of scales (up to 16 rows)
    static constexpr int kWBytes = kDecStageRows * CB * 16;   // packed words: [16 rows][CB][4 words]
    static constexpr int kSBytes = kDecStageRows * CB * 2;    // up to 16 rows of group scales (G = 32)
    static constexpr int kRedBytes = kConsumers * MR * kWarpCols * 4;  // per-warp sums, over the weight ring
    static constexpr int kMaxSmem = kDecSmemBudget + 3 * kDecMaxRing * 8 + 16 + 128;
    static_assert(kRedBytes <= 2 * kWBytes, "the final reduction fits in a weight ring of two slots");
    static_assert(CB % kBoxCols == 0 && kBoxCols * 4 <= 256, "weight boxes of at most 256 words");
    // byte offset of 16-column sub-block sb of a warp's columns in a slot's words, and
    // of its scales (in halves) from the warp's first column
    __host__ __device__ static constexpr int sb_words(int sb) { return (16 * sb / kBoxCols) * kBoxBytes + (16 * sb % kBoxCols) * 16; }
    __host__ __device__ static constexpr int sb_scales(int sb) { return kNarrowBoxes ? sb * kSBoxHalves : 16 * sb; }
};

// d = a * b (the accumulator starts from zero)
__device__ __forceinline__ void mma_16816_zero(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

// d += a * b
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// The eight codes of one packed word as four exact FP16 pairs of (q - 8): pairs
// (k, k+1), (k+2, k+3), (k+4, k+5), (k+6, k+7) from nibbles (0,4), (1,5), (2,6), (3,7).
// A low nibble OR-ed into the mantissa of 1024.0 gives 1024 + q, a high nibble
// 1024 + 16q (the ulp at 1024 is 1); 1024 + q - 1032 and (1024 + 16q)/16 - 72 are
// q - 8 exactly.
__device__ __forceinline__ void unpack_q8(uint32_t w, uint32_t (&o)[4])
{
    const uint32_t lo = 0x000F000Fu, hi = 0x00F000F0u, magic = 0x64006400u;
    const __half2 c1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
    const __half2 c1_16 = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
    const __half2 cm72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));
    const uint32_t w8 = w >> 8;
    const uint32_t a = and_or(w, lo, magic), b = and_or(w, hi, magic);
    const uint32_t c = and_or(w8, lo, magic), d = and_or(w8, hi, magic);
    const __half2 ha = __hsub2(u32_as_half2(a), c1032);
    const __half2 hb = __hfma2(u32_as_half2(b), c1_16, cm72);
    const __half2 hc = __hsub2(u32_as_half2(c), c1032);
    const __half2 hd = __hfma2(u32_as_half2(d), c1_16, cm72);
    o[0] = *reinterpret_cast<const uint32_t*>(&ha);
    o[1] = *reinterpret_cast<const uint32_t*>(&hb);
    o[2] = *reinterpret_cast<const uint32_t*>(&hc);
    o[3] = *reinterpret_cast<const uint32_t*>(&hd);
}

template <int MR, int CB, bool EPI>
__global__ void __launch_bounds__(kDecThreads, 2) w4a16_decode_kernel(const __grid_constant__ CUtensorMap tmap_w,
                                                                     const __grid_constant__ CUtensorMap tmap_s,
                                                                     const __grid_constant__ CUtensorMap tmap_x,
                                                                     const DecodeParams p)
{
    using C = DecCfg<MR, CB>;
    constexpr int NSB = C::kWarpCols / 16;   // 16-column sub-blocks of a consumer warp
    constexpr int NH = MR / 8;     // 8-row halves of X
    constexpr int KC = NSB >= 4 ? 1 : 4 / NSB;   // independent accumulators per sub-block in a full stage
    constexpr bool kFullPath = MR == 8 || NSB == 1;  // sixteen rows over 32+ columns keep the generic loop (registers)
    const int S = p.ring;
    const int xb = kDecStageRows * p.x_rows * 64;   // X bytes of a slot
    const int off_s = S * C::kWBytes;
    const int off_x = off_s + S * C::kSBytes;
    const int off_bar = off_x + S * xb;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((128 - (smem_addr(smem_raw) & 127)) & 127);
    const uint32_t sbase = smem_addr(smem);
    // wfull: the stage's words and scales landed (one arrival, with their bytes);
    // xfull: its X landed; empty: every consumer warp is done with the slot
    auto wfull_bar = [&](int s) { return sbase + off_bar + 8u * s; };
    auto xfull_bar = [&](int s) { return sbase + off_bar + 8u * (kDecMaxRing + s); };
    auto empty_bar = [&](int s) { return sbase + off_bar + 8u * (2 * kDecMaxRing + s); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + off_bar + 3 * kDecMaxRing * 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(wfull_bar(s), 1);
            mbar_init(xfull_bar(s), 1);
            mbar_init(empty_bar(s), C::kColTeams ? kConsumers : kConsumers / 2);   // the warps that take the stage
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // The next kernel may be scheduled now; it waits for this one before it reads
    // anything this one writes.
    if (threadIdx.x == 0) launch_dependents();
    const WaitCtl ctl{abort_flag, p.status, p.wait_limit_ns};
    const int n0 = blockIdx.x * CB;
    const int nt = n0 >> 7;

    if (warp == kProdW || warp == kProdX) {
        // ------------------------------------------------------------ producers
        // Packed words and scales: no earlier kernel in the stream writes them, so
        // they stream at once. X may be the previous kernel's output: its producer
        // waits for that kernel to complete first.
        const bool is_x = warp == kProdX;
        if (is_x) wait_prior_grid();
        if (lane == 0) {
            if (is_x) {
                prefetch_tmap(&tmap_x);
            } else {
                prefetch_tmap(&tmap_w);
                prefetch_tmap(&tmap_s);
            }
        }
        const uint32_t w_tx = (uint32_t)(C::kWBytes + p.scale_rows * CB * 2);
        int st = 0, s = 0;
        uint32_t ph = 0;   // phase of slot s: stage st uses slot st mod S in phase (st / S) mod 2
        for (; st < p.stages; ++st, s = s + 1 == S ? 0 : s + 1, ph ^= s == 0) {
            if (__any_sync(0xffffffffu, *abort_flag != 0) || !wait_warp<true>(empty_bar(s), ph ^ 1, ctl)) break;
            if (lane == 0) {
                if (is_x) {
                    mbar_arrive_expect_tx(xfull_bar(s), (uint32_t)xb);
                    tma_load_3d(sbase + off_x + s * xb, &tmap_x, xfull_bar(s), 0, 0, st * kDecStageRows);
                } else {
                    const int g0 = min((st * kDecStageRows * 32) >> p.g_shift, p.ng - 1);
                    mbar_arrive_expect_tx(wfull_bar(s), w_tx);
#pragma unroll
                    for (int bx = 0; bx < CB / C::kBoxCols; ++bx) {
                        const int col = n0 + bx * C::kBoxCols;   // the box's first column: one tile holds it
                        tma_load_2d(sbase + s * C::kWBytes + bx * C::kBoxBytes, &tmap_w, wfull_bar(s),
                                    (col & 127) * 4, (col >> 7) * p.tile_rows + st * kDecStageRows);
                        if constexpr (C::kNarrowBoxes)
                            tma_load_2d(sbase + off_s + s * C::kSBytes + bx * C::kSBoxHalves * 2, &tmap_s,
                                        wfull_bar(s), col & 127, (col >> 7) * p.ng + g0);
                    }
                    if constexpr (!C::kNarrowBoxes)
                        tma_load_2d(sbase + off_s + s * C::kSBytes, &tmap_s, wfull_bar(s), n0 & 127, nt * p.ng + g0);
                }
            }
            __syncwarp();
        }
        // Wind down: the copies in flight land before the CTA can exit (a full
        // barrier depends on its producer's arrival and the copies alone).
        if (lane == 0) {
            const int inflight = st < S ? st : S;
            for (int k = 1; k <= inflight; ++k) {
                const int q = st - k;
                wait_drain(is_x ? xfull_bar(q % S) : wfull_bar(q % S), (uint32_t)(q / S) & 1, 1000000000LL);
            }
        }
    } else {
        // ------------------------------------------------------------ consumers
        // The residual may be the previous kernel's output, and Y may still be read by it.
        wait_prior_grid();
        const int g = lane >> 2, t = lane & 3;
        // Two teams of four warps take the stages in turn (or, with 128-column blocks,
        // every stage for their own 64 columns); warp wl of a team takes rows
        // 4wl .. 4wl+3 of a stage (128 values of k: one group when G >= 128).
        const int team = warp >> 2, wl = warp & 3;
        const int cbase = C::kColTeams ? team * C::kWarpCols : 0;   // the warp's first column in the block
        constexpr int kStep = C::kColTeams ? 1 : 2;                  // stages between two of a warp's stages
        const int rpg = p.g_shift >= 7 ? 4 : 1 << (p.g_shift - 5);   // rows per group: 4, 2 (G = 64) or 1 (G = 32)
        // lane offsets: X rows g and 8 + g (lanes past the last row of X read the last
        // row again, for output columns that are never stored), the warp's words
        int xoff[NH];
#pragma unroll
        for (int h = 0; h < NH; ++h) xoff[h] = min(8 * h + g, p.x_rows - 1) * 64 + t * 16;
        const int woff = (cbase / C::kBoxCols) * C::kBoxBytes + (4 * wl * C::kBoxCols + cbase % C::kBoxCols + g) * 16 + t * 4;
        float acc[NSB][NH][4];
#pragma unroll
        for (int sb = 0; sb < NSB; ++sb)
#pragma unroll
            for (int h = 0; h < NH; ++h)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[sb][h][e] = 0.f;
        bool ok = true;
        int s = C::kColTeams ? 0 : team;   // slot of stage st; S >= 2
        uint32_t ph = 0;
        // With the teams taking stages in turn and an odd ring, stages st and st + S
        // share a slot but go to different teams: a team first waits until the slot's
        // earlier stage is consumed (the producer's own wait), so that it never waits
        // on the full barriers two phases ahead, where the parity of the earlier phase
        // would pass for the later one.
        const bool odd_ring = !C::kColTeams && (S & 1);
        for (int st = C::kColTeams ? 0 : team; st < p.stages; st += kStep) {
            if (odd_ring && !wait_warp<true>(empty_bar(s), ph ^ 1, ctl)) {
                ok = false;
                break;
            }
            if (!wait_warp<true>(wfull_bar(s), ph, ctl) || !wait_warp<true>(xfull_bar(s), ph, ctl)) {
                ok = false;
                break;
            }
            const int g0 = min((st * kDecStageRows * 32) >> p.g_shift, p.ng - 1);
            if (kFullPath && rpg == 4 && (st + 1) * kDecStageRows <= p.rows) {
                // A full stage with G >= 128: the warp's four rows are 128 values of k
                // of one group. No guard between the rows, so their loads can be issued
                // together; with fewer than four sub-blocks the rows go to independent
                // accumulators (KC chains) that are added before the scale.
                float ch[KC][NSB][NH][4];
                const uint8_t* xs = smem + off_x + s * xb + 4 * wl * p.x_rows * 64;
                const uint8_t* ws = smem + s * C::kWBytes + woff;
#pragma unroll
                for (int rr = 0; rr < 4; ++rr) {
                    uint4 xv[NH];
#pragma unroll
                    for (int h = 0; h < NH; ++h)
                        xv[h] = *reinterpret_cast<const uint4*>(xs + rr * p.x_rows * 64 + xoff[h]);
                    const uint8_t* wa = ws + rr * C::kBoxCols * 16;
#pragma unroll
                    for (int sb = 0; sb < NSB; ++sb) {
                        uint32_t pa[4], pb[4];
                        unpack_q8(*reinterpret_cast<const uint32_t*>(wa + C::sb_words(sb)), pa);
                        unpack_q8(*reinterpret_cast<const uint32_t*>(wa + C::sb_words(sb) + 128), pb);
                        const uint32_t a1[4] = {pa[0], pb[0], pa[1], pb[1]};
                        const uint32_t a2[4] = {pa[2], pb[2], pa[3], pb[3]};
#pragma unroll
                        for (int h = 0; h < NH; ++h) {
                            if (rr < KC)
                                mma_16816_zero(ch[rr % KC][sb][h], a1, xv[h].x, xv[h].y);
                            else
                                mma_16816(ch[rr % KC][sb][h], a1, xv[h].x, xv[h].y);
                            mma_16816(ch[rr % KC][sb][h], a2, xv[h].z, xv[h].w);
                        }
                    }
                }
                const int gl = ((st * kDecStageRows + 4 * wl) * 32 >> p.g_shift) - g0;
                const __half* sc = reinterpret_cast<const __half*>(smem + off_s + s * C::kSBytes) +
                                   (C::kNarrowBoxes ? gl * 16 : gl * CB + cbase) + g;
#pragma unroll
                for (int sb = 0; sb < NSB; ++sb) {
                    const float s_lo = __half2float(sc[C::sb_scales(sb)]), s_hi = __half2float(sc[C::sb_scales(sb) + 8]);
#pragma unroll
                    for (int h = 0; h < NH; ++h) {
#pragma unroll
                        for (int c = 1; c < KC; ++c)
#pragma unroll
                            for (int e = 0; e < 4; ++e) ch[0][sb][h][e] += ch[c][sb][h][e];
                        acc[sb][h][0] = fmaf(s_lo, ch[0][sb][h][0], acc[sb][h][0]);
                        acc[sb][h][1] = fmaf(s_lo, ch[0][sb][h][1], acc[sb][h][1]);
                        acc[sb][h][2] = fmaf(s_hi, ch[0][sb][h][2], acc[sb][h][2]);
                        acc[sb][h][3] = fmaf(s_hi, ch[0][sb][h][3], acc[sb][h][3]);
                    }
                }
            } else {
            // sums of the current group: the first MMA of a group starts from zero
            float gacc[NSB][NH][4];
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) {
                const int rl = 4 * wl + rr;                   // row within the stage
                const int row = st * kDecStageRows + rl;      // row of 32 values of k
                if (row < p.rows) {
                    // rows g and 8 + g of X; lanes past the last row read the last row
                    // again, for output columns that are never stored
                    const uint8_t* xa = smem + off_x + s * xb + rl * p.x_rows * 64;
                    uint4 xv[NH];
#pragma unroll
                    for (int h = 0; h < NH; ++h) xv[h] = *reinterpret_cast<const uint4*>(xa + xoff[h]);
                    // the box of the warp's columns; within it column 16 sb + g (and + 8) of row rl
                    const uint8_t* wa = smem + s * C::kWBytes + (cbase / C::kBoxCols) * C::kBoxBytes +
                                        (rl * C::kBoxCols + cbase % C::kBoxCols + g) * 16 + t * 4;
                    const bool first = (rr & (rpg - 1)) == 0;
#pragma unroll
                    for (int sb = 0; sb < NSB; ++sb) {
                        uint32_t pa[4], pb[4];
                        unpack_q8(*reinterpret_cast<const uint32_t*>(wa + C::sb_words(sb)), pa);         // column 16 sb + g
                        unpack_q8(*reinterpret_cast<const uint32_t*>(wa + C::sb_words(sb) + 128), pb);   // column 16 sb + g + 8
                        const uint32_t a1[4] = {pa[0], pb[0], pa[1], pb[1]};
                        const uint32_t a2[4] = {pa[2], pb[2], pa[3], pb[3]};
#pragma unroll
                        for (int h = 0; h < NH; ++h) {
                            if (first)
                                mma_16816_zero(gacc[sb][h], a1, xv[h].x, xv[h].y);
                            else
                                mma_16816(gacc[sb][h], a1, xv[h].x, xv[h].y);
                            mma_16816(gacc[sb][h], a2, xv[h].z, xv[h].w);
                        }
                    }
                    if (((rr + 1) & (rpg - 1)) == 0 || row + 1 == p.rows) {
                        // the group's sums, times the scales of columns g and g + 8 of
                        // each sub-block, go to the running sums
                        const int gl = min((row * 32) >> p.g_shift, p.ng - 1) - g0;
                        const __half* sc = reinterpret_cast<const __half*>(smem + off_s + s * C::kSBytes) +
                                           (C::kNarrowBoxes ? gl * 16 : gl * CB + cbase) + g;
#pragma unroll
                        for (int sb = 0; sb < NSB; ++sb) {
                            const float s_lo = __half2float(sc[C::sb_scales(sb)]),
                                        s_hi = __half2float(sc[C::sb_scales(sb) + 8]);
#pragma unroll
                            for (int h = 0; h < NH; ++h) {
                                acc[sb][h][0] = fmaf(s_lo, gacc[sb][h][0], acc[sb][h][0]);
                                acc[sb][h][1] = fmaf(s_lo, gacc[sb][h][1], acc[sb][h][1]);
                                acc[sb][h][2] = fmaf(s_hi, gacc[sb][h][2], acc[sb][h][2]);
                                acc[sb][h][3] = fmaf(s_hi, gacc[sb][h][3], acc[sb][h][3]);
                            }
                        }
                    }
                }
            }
            }
            fence_proxy_async_smem();   // the loads of the slot precede its next TMA copies
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(s));
            s += kStep;
            if (s >= S) {
                s -= S;
                ph ^= 1;
            }
        }

        // Every consumer is done with the ring (or gave up): the weight ring holds
        // the warps' sums, [warp][MR][the warp's columns], added in warp order over
        // the warps that hold a column (all eight, or the four of its team).
        constexpr int WC = C::kWarpCols;
        named_bar_sync(1, 32 * kConsumers);
        float* red = reinterpret_cast<float*>(smem);
        if (ok) {
#pragma unroll
            for (int sb = 0; sb < NSB; ++sb)
#pragma unroll
                for (int h = 0; h < NH; ++h) {
                    const int m = 8 * h + 2 * t, c = 16 * sb + g;
                    float* r = red + (warp * MR + m) * WC + c;
                    r[0] = acc[sb][h][0];
                    r[WC] = acc[sb][h][1];
                    r[8] = acc[sb][h][2];
                    r[WC + 8] = acc[sb][h][3];
                }
        }
        named_bar_sync(1, 32 * kConsumers);
        if (!*abort_flag) {
            for (int i = threadIdx.x; i < MR * CB; i += 32 * kConsumers) {
                const int m = i / CB, c = i % CB, n = n0 + c;
                if (m < p.M && n < p.N) {
                    float v = 0.f;
                    if constexpr (C::kColTeams) {
                        const int tm = c / WC, cl = c % WC;
#pragma unroll
                        for (int w = 0; w < kConsumers / 2; ++w) v += red[((tm * 4 + w) * MR + m) * WC + cl];
                    } else {
#pragma unroll
                        for (int w = 0; w < kConsumers; ++w) v += red[(w * MR + m) * WC + c];
                    }
                    if constexpr (EPI)
                        v = epilogue_op(p.act, v, ld16<false>(p.bias, n), ld16<false>(p.residual, (size_t)m * p.ldr + n));
                    p.y[(size_t)m * p.ldy + n] = __float2half_rn(v);
                }
            }
        }
    }
}

template <int MR, int CB, bool EPI>
cudaError_t setup_one()
{
    return cudaFuncSetAttribute(w4a16_decode_kernel<MR, CB, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                DecCfg<MR, CB>::kMaxSmem);
}

template <int MR, int CB>
cudaError_t launch_one(const CUtensorMap& tw, const CUtensorMap& ts, const CUtensorMap& tx, const DecodeParams& p,
                       bool epi, int grid, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kDecThreads);
    cfg.dynamicSmemBytes = decode_smem_bytes(CB, p.x_rows, p.ring);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return epi ? cudaLaunchKernelEx(&cfg, w4a16_decode_kernel<MR, CB, true>, tw, ts, tx, p)
               : cudaLaunchKernelEx(&cfg, w4a16_decode_kernel<MR, CB, false>, tw, ts, tx, p);
}

template <int MR>
cudaError_t launch_mr(const CUtensorMap& tw, const CUtensorMap& ts, const CUtensorMap& tx, const DecodeParams& p,
                      int cb, bool epi, int grid, cudaStream_t stream)
{
    switch (cb) {
        case 16: return launch_one<MR, 16>(tw, ts, tx, p, epi, grid, stream);
        case 32: return launch_one<MR, 32>(tw, ts, tx, p, epi, grid, stream);
        case 48:
            if constexpr (MR == 8) return launch_one<MR, 48>(tw, ts, tx, p, epi, grid, stream);
            return cudaErrorInvalidValue;
        case 64: return launch_one<MR, 64>(tw, ts, tx, p, epi, grid, stream);
        case 80:
            if constexpr (MR == 8) return launch_one<MR, 80>(tw, ts, tx, p, epi, grid, stream);
            return cudaErrorInvalidValue;
        case 128: return launch_one<MR, 128>(tw, ts, tx, p, epi, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int MR>
cudaError_t setup_mr()
{
    cudaError_t e;
    if ((e = setup_one<MR, 16, false>()) != cudaSuccess || (e = setup_one<MR, 16, true>()) != cudaSuccess ||
        (e = setup_one<MR, 32, false>()) != cudaSuccess || (e = setup_one<MR, 32, true>()) != cudaSuccess ||
        (e = setup_one<MR, 64, false>()) != cudaSuccess || (e = setup_one<MR, 64, true>()) != cudaSuccess ||
        (e = setup_one<MR, 128, false>()) != cudaSuccess || (e = setup_one<MR, 128, true>()) != cudaSuccess)
        return e;
    if constexpr (MR == 8) {
        if ((e = setup_one<MR, 48, false>()) != cudaSuccess || (e = setup_one<MR, 48, true>()) != cudaSuccess ||
            (e = setup_one<MR, 80, false>()) != cudaSuccess || (e = setup_one<MR, 80, true>()) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

}  // namespace

cudaError_t setup_decode()
{
    cudaError_t e;
    if ((e = setup_mr<8>()) != cudaSuccess || (e = setup_mr<16>()) != cudaSuccess) return e;
    return cudaSuccess;
}

cudaError_t launch_decode(const CUtensorMap& tmap_w, const CUtensorMap& tmap_s, const CUtensorMap& tmap_x,
                          const DecodeParams& p, int mr, int cb, bool epi, int grid, cudaStream_t stream)
{
    switch (mr) {
        case 8: return launch_mr<8>(tmap_w, tmap_s, tmap_x, p, cb, epi, grid, stream);
        case 16: return launch_mr<16>(tmap_w, tmap_s, tmap_x, p, cb, epi, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace w4a16
