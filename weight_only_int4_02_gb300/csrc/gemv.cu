// W4A16 matmul for one to four rows of X on the CUDA cores (no tensor cores, no
// tensor memory, no split-K workspace).
//
// Y[m][n] = sum_g s[g][n] * sum_{k in g} X[m][k] * (q[k][n] - 8), FP32 accumulate, FP16 out.
//
// With one to four rows of X the matmul is a handful of dot products per weight
// column: every packed weight is read once from HBM and used M times, so the
// kernel is a stream of the packed words with as little arithmetic per weight as
// the unpack allows. It reads the same packed layout (version 2) and tile-ordered
// scales as the tensor-core kernel, so one packed buffer serves both paths.
//
// Work split: the output columns are cut into blocks of CB = 8 * CPT adjacent
// columns (16 or 32); a block is processed over the whole of K by one CTA (CTAs
// take blocks in turn), so no partial sum leaves the CTA and there is no global
// reduction. The reduction dimension is cut into rows of 32 values of k (one
// 16-byte unit of the packed layout per column) and stages of 32 rows.
//
// Roles: one producer warp streams the stages with TMA into a ring of four
// (the block's 32 rows x CB columns of packed words, one 2-D copy, and the
// stage's group scales, another); one converter warp turns the stage's 1024
// values of each row of X into FP32 in the same ring slot (every value once, for
// all the CTA's threads); eight consumer warps compute. The producer needs nothing
// from the previous kernel, so it fills the ring while that kernel is still
// running (programmatic dependent launch); the converter and the consumers wait
// for the previous kernel (griddepcontrol.wait) before they read X or write Y.
// Consumer lane l of warp w takes row 4w + l/8 of every stage and columns
// (l % 8) + 8j, j < CPT.
//
// Per row a thread turns each packed word into eight exact FP32 values
// (q - 8)/16: one LOP3 per nibble ORs the nibble, where it lies, into the
// mantissa of a power of two chosen for that bit position so that one unit of the
// nibble is worth 1/16 (2^19 for bits 0..3, 2^15 for bits 4..7, ... 2^3 for
// bits 16..19; the top three nibbles are shifted down by 12 first); a paired FP32
// subtraction of (power + 8/16) is exact (Sterbenz). The FP16 activations of the
// row are read as FP32 pairs and used for all of the thread's columns; paired
// FP32 fused multiply-adds (products of at most 15 significant bits, exact) sum
// the row's 32 terms per column and row of X, and the row sum is scaled once by
// 16 times the group's scale (a row never straddles two groups: G is 32, 64, 128
// or one group). Partials of a column are combined in a fixed order, across the
// lanes of a warp by shuffles and across warps through shared memory, so results
// are bit-identical from run to run.
//
// Every wait is bounded: a wait that runs out sets the CTA's abort flag and the
// library's error word for this kernel (read by w4a16_check_device_status); the
// consumers then skip the remaining rows, the producer stops issuing, waits
// (bounded) for its copies in flight, and the CTA returns.
//
// Sources: "quant_marlin_kernel" (aicassindra.com), "The architecture: every
// piece explained" (packed INT4, group scales, register-level unpack with bit
// operations and a lookup trick, FP16 activations in and out); "Low-Precision
// Quantization Kernels in Production" (llms.blog), section 2 (ExLlamaV2: the
// activation vector at batch 1 to 4, weights streamed, unpacked in registers,
// group-scaled and reduced across the threads of a warp) and section 5
// ("Decoding Roofline Dynamics": at batch 1 the matmul is a memory-bound GEMV).
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_tc.cuh"
#include "gemv.cuh"

namespace w4a16 {

namespace {

constexpr int kConsumerWarps = kGemvThreads / 32 - 2;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kConverterWarp = kConsumerWarps + 1;
constexpr int kStageRows = kGemvStageK / 32;   // rows of 32 k per stage
constexpr int kStages = 4;                     // ring depth
constexpr int kRowGroups = 4;                  // rows of a stage per consumer warp (lanes / 8)
static_assert(kConsumerWarps * kRowGroups == kStageRows, "one stage row per consumer thread");

template <int MR, int CPT>
struct GemvCfg {
    static constexpr int CB = 8 * CPT;                        // columns per block
    static constexpr int kWBytes = kStageRows * CB * 16;      // packed words of a stage
    static constexpr int kSBytes = kStageRows * CB * 2;       // up to 32 rows of group scales
    static constexpr int kXBytes = MR * kGemvStageK * 4;      // the stage's X in FP32, [MR][1024]
    static constexpr int kOffS = kStages * kWBytes;
    static constexpr int kOffX = kOffS + kStages * kSBytes;
    static constexpr int kOffBar = kOffX + kStages * kXBytes;
    static constexpr int kOffMisc = kOffBar + 3 * kStages * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 128;    // + alignment slack
};

// Activations: read by every CTA, kept in L1.
__device__ __forceinline__ uint4 ld_x16(const __half* p)
{
    uint4 v;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// The binary32 power of two 2^e with a zero mantissa.
__host__ __device__ constexpr uint32_t pow2_bits(int e) { return (uint32_t)(127 + e) << 23; }

// The eight codes of one packed word as exact FP32 (q - 8)/16, in four pairs in
// the order of k. Nibble i holds k0 + 2*(i%4) + i/4, so the pairs (k0, k0+1),
// (k0+2, k0+3), (k0+4, k0+5), (k0+6, k0+7) are nibbles (0,4), (1,5), (2,6), (3,7).
// Nibbles 0..4 are used where they lie (bits 4i..4i+3); nibbles 5, 6, 7 after a
// shift by 12 (bits 8..19). A nibble at bits b..b+3 OR-ed into the mantissa of
// 2^(19 - b) is worth q/16; subtracting 2^(19 - b) + 1/2 leaves (q - 8)/16 exactly.
__device__ __forceinline__ void unpack_word_f32(uint32_t w, float2 (&v)[4])
{
    const uint32_t u = w >> 12;
    const float2 a0 = make_float2(__uint_as_float(and_or(w, 0x0000000Fu, pow2_bits(19))),
                                  __uint_as_float(and_or(w, 0x000F0000u, pow2_bits(3))));
    const float2 a1 = make_float2(__uint_as_float(and_or(w, 0x000000F0u, pow2_bits(15))),
                                  __uint_as_float(and_or(u, 0x00000F00u, pow2_bits(11))));
    const float2 a2 = make_float2(__uint_as_float(and_or(w, 0x00000F00u, pow2_bits(11))),
                                  __uint_as_float(and_or(u, 0x0000F000u, pow2_bits(7))));
    const float2 a3 = make_float2(__uint_as_float(and_or(w, 0x0000F000u, pow2_bits(7))),
                                  __uint_as_float(and_or(u, 0x000F0000u, pow2_bits(3))));
    v[0] = __fadd2_rn(a0, make_float2(-(524288.f + 0.5f), -(8.f + 0.5f)));
    v[1] = __fadd2_rn(a1, make_float2(-(32768.f + 0.5f), -(2048.f + 0.5f)));
    v[2] = __fadd2_rn(a2, make_float2(-(2048.f + 0.5f), -(128.f + 0.5f)));
    v[3] = __fadd2_rn(a3, make_float2(-(128.f + 0.5f), -(8.f + 0.5f)));
}

template <int MR, int CPT, bool EPI>
__global__ void __launch_bounds__(kGemvThreads) w4a16_gemv_kernel(const __grid_constant__ CUtensorMap tmap_w,
                                                                  const __grid_constant__ CUtensorMap tmap_s,
                                                                  const GemvParams p)
{
    using C = GemvCfg<MR, CPT>;
    constexpr int CB = C::CB;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((128 - (smem_addr(smem_raw) & 127)) & 127);
    const uint32_t sbase = smem_addr(smem);
    // full: the stage's copies landed (one arrival, with their bytes); xready: the
    // converter wrote the stage's X; empty: every consumer warp is done with the slot
    auto full_bar = [&](int s) { return sbase + C::kOffBar + 8u * s; };
    auto empty_bar = [&](int s) { return sbase + C::kOffBar + 8u * (kStages + s); };
    auto xready_bar = [&](int s) { return sbase + C::kOffBar + 8u * (2 * kStages + s); };
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc);
    __shared__ float red[kConsumerWarps][MR][CB];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(full_bar(s), 1);                 // producer, with the copies' bytes
            mbar_init(xready_bar(s), 1);               // converter
            mbar_init(empty_bar(s), kConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // The next kernel may be scheduled now; it waits for this one before it reads
    // anything this one writes.
    if (threadIdx.x == 0) launch_dependents();
    const WaitCtl ctl{abort_flag, p.status, p.wait_limit_ns};

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        // Packed weights and scales only: no earlier kernel in the stream writes
        // them, so the ring fills before the previous kernel has finished.
        if (lane == 0) {
            prefetch_tmap(&tmap_w);
            prefetch_tmap(&tmap_s);
        }
        uint32_t seq = 0;
        bool ok = true;
        const uint32_t stage_tx = (uint32_t)(C::kWBytes + p.scale_rows * CB * 2);
        for (int b = blockIdx.x; ok && b < p.blocks; b += gridDim.x) {
            const int n0 = b * CB;
            const int nt = n0 >> 7;
            for (int st = 0; st < p.stages; ++st, ++seq) {
                const int s = (int)(seq % kStages);
                if (__any_sync(0xffffffffu, *abort_flag != 0) || !wait_warp<true>(empty_bar(s), ((seq / kStages) & 1) ^ 1, ctl)) {
                    ok = false;
                    break;
                }
                if (lane == 0) {
                    const int g0 = min((st * kGemvStageK) >> p.g_shift, p.ng - 1);
                    mbar_arrive_expect_tx(full_bar(s), stage_tx);
                    tma_load_2d(sbase + s * C::kWBytes, &tmap_w, full_bar(s), (n0 & 127) * 4,
                                nt * p.tile_rows + st * kStageRows);
                    tma_load_2d(sbase + C::kOffS + s * C::kSBytes, &tmap_s, full_bar(s), n0 & 127, nt * p.ng + g0);
                }
                __syncwarp();
            }
        }
        // Wind down: let the copies in flight land before the CTA can exit (the full
        // barriers depend on the copies alone).
        if (lane == 0) {
            const uint32_t inflight = seq < (uint32_t)kStages ? seq : (uint32_t)kStages;
            for (uint32_t k = 1; k <= inflight; ++k) {
                const uint32_t q = seq - k;
                wait_drain(full_bar((int)(q % kStages)), (q / kStages) & 1, 1000000000LL);
            }
        }
    } else if (warp == kConverterWarp) {
        // ------------------------------------------------------------ converter
        // X may be the previous kernel's output. Each stage's 1024 values of every
        // row of X become FP32 in the stage's slot (zero past K and past M).
        wait_prior_grid();
        uint32_t seq = 0;
        for (int b = blockIdx.x; b < p.blocks; b += gridDim.x) {
            for (int st = 0; st < p.stages; ++st, ++seq) {
                const int s = (int)(seq % kStages);
                if (__any_sync(0xffffffffu, *abort_flag != 0) || !wait_warp<true>(empty_bar(s), ((seq / kStages) & 1) ^ 1, ctl)) break;
                float* xs = reinterpret_cast<float*>(smem + C::kOffX + s * C::kXBytes);
#pragma unroll
                for (int m = 0; m < MR; ++m) {
#pragma unroll
                    for (int q = 0; q < kGemvStageK / 256; ++q) {
                        const int kl = q * 256 + lane * 8;     // 8 values of k per lane and step
                        const int k = st * kGemvStageK + kl;
                        float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
                        if (m < p.M && k < p.K) {
                            const uint4 xv = ld_x16(p.x + (size_t)m * p.ldx + k);
                            const float2 a = __half22float2(u32_as_half2(xv.x)), b2 = __half22float2(u32_as_half2(xv.y));
                            const float2 c = __half22float2(u32_as_half2(xv.z)), d = __half22float2(u32_as_half2(xv.w));
                            lo = make_float4(a.x, a.y, b2.x, b2.y);
                            hi = make_float4(c.x, c.y, d.x, d.y);
                        }
                        *reinterpret_cast<float4*>(xs + m * kGemvStageK + kl) = lo;
                        *reinterpret_cast<float4*>(xs + m * kGemvStageK + kl + 4) = hi;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(xready_bar(s));   // release: the writes above precede the arrival
            }
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        }
    } else {
        // ------------------------------------------------------------ consumers
        // The residual may be the previous kernel's output, and Y may still be read
        // by it.
        wait_prior_grid();
        const int cl = lane & 7;
        const int row_in_stage = warp * kRowGroups + (lane >> 3);
        uint32_t seq = 0;
        bool ok = true;
        for (int b = blockIdx.x; b < p.blocks; b += gridDim.x) {
            float acc[CPT][MR];
#pragma unroll
            for (int j = 0; j < CPT; ++j)
#pragma unroll
                for (int m = 0; m < MR; ++m) acc[j][m] = 0.f;
            for (int st = 0; st < p.stages; ++st, ++seq) {
                if (!ok) continue;
                const int s = (int)(seq % kStages);
                if (!wait_warp<true>(full_bar(s), (seq / kStages) & 1, ctl) ||
                    !wait_warp<true>(xready_bar(s), (seq / kStages) & 1, ctl)) {
                    ok = false;
                    continue;
                }
                const int r = st * kStageRows + row_in_stage;
                if (r < p.rows) {
                    const uint8_t* wrow = smem + s * C::kWBytes + row_in_stage * CB * 16 + cl * 16;
                    uint4 wv[CPT];
#pragma unroll
                    for (int j = 0; j < CPT; ++j) wv[j] = *reinterpret_cast<const uint4*>(wrow + j * 128);
                    const int g0 = min((st * kGemvStageK) >> p.g_shift, p.ng - 1);
                    const int g = min((r * 32) >> p.g_shift, p.ng - 1);
                    const __half* srow = reinterpret_cast<const __half*>(smem + C::kOffS + s * C::kSBytes) +
                                         (g - g0) * CB + cl;
                    float sc[CPT];
#pragma unroll
                    for (int j = 0; j < CPT; ++j) sc[j] = 16.f * __half2float(srow[8 * j]);
                    float2 pa[CPT][MR];
#pragma unroll
                    for (int j = 0; j < CPT; ++j)
#pragma unroll
                        for (int m = 0; m < MR; ++m) pa[j][m] = make_float2(0.f, 0.f);
#pragma unroll
                    for (int wd = 0; wd < 4; ++wd) {
                        const int kk = r * 32 + 8 * wd;
                        if (kk >= p.K) break;   // K is a multiple of 8: a word is all in or all out
                        float2 xf[MR][4];
#pragma unroll
                        for (int m = 0; m < MR; ++m) {
                            const float4* xs = reinterpret_cast<const float4*>(
                                smem + C::kOffX + s * C::kXBytes + (m * kGemvStageK + row_in_stage * 32 + 8 * wd) * 4);
                            const float4 lo = xs[0], hi = xs[1];
                            xf[m][0] = make_float2(lo.x, lo.y);
                            xf[m][1] = make_float2(lo.z, lo.w);
                            xf[m][2] = make_float2(hi.x, hi.y);
                            xf[m][3] = make_float2(hi.z, hi.w);
                        }
#pragma unroll
                        for (int j = 0; j < CPT; ++j) {
                            const uint32_t word = wd == 0 ? wv[j].x : wd == 1 ? wv[j].y : wd == 2 ? wv[j].z : wv[j].w;
                            float2 v[4];
                            unpack_word_f32(word, v);
#pragma unroll
                            for (int m = 0; m < MR; ++m)
#pragma unroll
                                for (int t = 0; t < 4; ++t) pa[j][m] = __ffma2_rn(v[t], xf[m][t], pa[j][m]);
                        }
                    }
#pragma unroll
                    for (int j = 0; j < CPT; ++j)
#pragma unroll
                        for (int m = 0; m < MR; ++m) acc[j][m] = fmaf(pa[j][m].x + pa[j][m].y, sc[j], acc[j][m]);
                }
                fence_proxy_async_smem();   // the loads of the slot precede its next TMA copies
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(s));
            }

            // Lanes cl, cl + 8, cl + 16, cl + 24 of a warp hold partials of the same columns.
#pragma unroll
            for (int off = 8; off <= 16; off <<= 1)
#pragma unroll
                for (int j = 0; j < CPT; ++j)
#pragma unroll
                    for (int m = 0; m < MR; ++m) acc[j][m] += __shfl_xor_sync(0xffffffffu, acc[j][m], off);
            if (lane < 8)
#pragma unroll
                for (int j = 0; j < CPT; ++j)
#pragma unroll
                    for (int m = 0; m < MR; ++m) red[warp][m][cl + 8 * j] = acc[j][m];
            named_bar_sync(1, 32 * kConsumerWarps);
            if (threadIdx.x < MR * CB) {
                const int m = threadIdx.x / CB, c = threadIdx.x % CB;
                const int nn = b * CB + c;
                float v = 0.f;
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) v += red[w][m][c];
                if (m < p.M && nn < p.N) {
                    if constexpr (EPI)
                        v = epilogue_op(p.act, v, ld16<false>(p.bias, nn), ld16<false>(p.residual, (size_t)m * p.ldr + nn));
                    p.y[(size_t)m * p.ldy + nn] = __float2half_rn(v);
                }
            }
            named_bar_sync(1, 32 * kConsumerWarps);
        }
    }
}

// CTAs of each instantiation one SM holds at once (filled in by setup_gemv).
int g_resident[3][2][2];   // [mr 1, 2, 4][cb 16, 32][epilogue]

int mr_index(int mr) { return mr == 1 ? 0 : mr == 2 ? 1 : 2; }

template <int MR, int CPT, bool EPI>
cudaError_t setup_one()
{
    auto kernel = w4a16_gemv_kernel<MR, CPT, EPI>;
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GemvCfg<MR, CPT>::kSmemBytes);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, kGemvThreads, GemvCfg<MR, CPT>::kSmemBytes);
    if (e != cudaSuccess) return e;
    g_resident[mr_index(MR)][CPT == 4 ? 1 : 0][EPI ? 1 : 0] = n > 0 ? n : 1;
    return cudaSuccess;
}

template <int MR, int CPT>
cudaError_t launch_one(const CUtensorMap& tw, const CUtensorMap& ts, const GemvParams& p, bool epi, int grid,
                       cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kGemvThreads);
    cfg.dynamicSmemBytes = GemvCfg<MR, CPT>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return epi ? cudaLaunchKernelEx(&cfg, w4a16_gemv_kernel<MR, CPT, true>, tw, ts, p)
               : cudaLaunchKernelEx(&cfg, w4a16_gemv_kernel<MR, CPT, false>, tw, ts, p);
}

template <int MR>
cudaError_t launch_cb(const CUtensorMap& tw, const CUtensorMap& ts, const GemvParams& p, int cb, bool epi, int grid,
                      cudaStream_t stream)
{
    switch (cb) {
        case 16: return launch_one<MR, 2>(tw, ts, p, epi, grid, stream);
        case 32: return launch_one<MR, 4>(tw, ts, p, epi, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int MR>
cudaError_t setup_mr()
{
    cudaError_t e;
    if ((e = setup_one<MR, 2, false>()) != cudaSuccess || (e = setup_one<MR, 2, true>()) != cudaSuccess ||
        (e = setup_one<MR, 4, false>()) != cudaSuccess || (e = setup_one<MR, 4, true>()) != cudaSuccess)
        return e;
    return cudaSuccess;
}

}  // namespace

cudaError_t setup_gemv()
{
    cudaError_t e;
    if ((e = setup_mr<1>()) != cudaSuccess || (e = setup_mr<2>()) != cudaSuccess || (e = setup_mr<4>()) != cudaSuccess)
        return e;
    return cudaSuccess;
}

int gemv_resident_ctas(int mr, int cb, bool epi) { return g_resident[mr_index(mr)][cb == 32 ? 1 : 0][epi ? 1 : 0]; }

cudaError_t launch_gemv(const CUtensorMap& tmap_w, const CUtensorMap& tmap_s, const GemvParams& p, int mr, int cb,
                        bool epi, int grid, cudaStream_t stream)
{
    switch (mr) {
        case 1: return launch_cb<1>(tmap_w, tmap_s, p, cb, epi, grid, stream);
        case 2: return launch_cb<2>(tmap_w, tmap_s, p, cb, epi, grid, stream);
        case 4: return launch_cb<4>(tmap_w, tmap_s, p, cb, epi, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace w4a16
