// W4A16 matmul on tcgen05 tensor cores, one persistent CTA per SM.
//
// Y[M][N] = X[M][K] * W[K][N], W[k][n] = (q - 8) * s[k/G][n], FP32 accumulate, FP16 out.
//
// The MMA runs "swapped": D[n][m] = sum_k W^T[n][k] * X^T[k][m], so the weight
// tile is the 128-row A operand and X supplies the N operand (tile_m rows of X,
// 16..256). A lives in tensor memory: dequant warps unpack the INT4 codes
// with bit operations (magic-number FP16 construction) straight into TMEM
// columns, so dequantised weights never touch shared memory; B (X) is loaded
// by TMA into 128-byte-swizzled shared memory; D accumulates in TMEM.
//
// Warp roles (448 threads):
//   warps 0-3   epilogue: TMEM -> registers -> FP16 Y, or FP32 partials + fix-up
//   warps 4-11  dequant: packed words (shared) -> FP16 (q-8)*s -> TMEM A ring
//   warp 12     producer: TMA X tile, bulk copy of packed words and scales
//   warp 13     MMA issuer (one thread) and TMEM owner
//
// Work split ("stream-K"): the iteration space (tile, 64-wide K chunk) is cut
// into one contiguous range per CTA. A tile whose chunks span several CTAs is
// reduced in global memory: every contributor stores its FP32 partial, and the
// last one to arrive on the tile's counter sums all partials in contributor
// order, so the result does not depend on arrival order.
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
constexpr int kChunkK = 64;        // K values per pipeline stage
constexpr int kChunkWords = 1024;  // packed words per (tile, chunk): 128 * 64 / 8
constexpr int kChunkBytes = 4096;
constexpr int kScaleSlotBytes = 512;  // up to two groups of 128 FP16 scales per chunk
constexpr int kThreads = 448;
constexpr int kAStages = 4;        // TMEM A ring depth (32 columns each)

struct GemmParams {
    const uint32_t* packed;
    const __half* scales;  // tile-ordered scales [n_tiles][ng][128]
    __half* y;
    float* partials;       // [2 * grid][tile_m][128] FP32
    int* counters;         // [grid], zero between launches
    int* status;           // error word, bit 0 = a wait timed out
    int M, N, K, G, ng;
    int n_tiles, m_tiles, KC;
    long long total_iters;  // n_tiles * m_tiles * KC
    int grid;
    long long wait_limit_ns;
};

template <int TM>
struct TcCfg {
    static constexpr int kXBytes = TM * 128;  // TM rows x 64 FP16
    static constexpr int kStageBytes = kXBytes + kChunkBytes + kScaleSlotBytes;
    static constexpr int kStagesRaw = (200 * 1024) / kStageBytes;
    static constexpr int kStages = kStagesRaw > 16 ? 16 : kStagesRaw;
    static constexpr int kDBufs = TM <= 128 ? 2 : 1;
    static constexpr int kACol = 0;
    static constexpr int kDCol = kAStages * 32;
    static constexpr int kColsUsed = kDCol + kDBufs * TM;
    static constexpr int kTmemCols = kColsUsed <= 256 ? 256 : 512;
    // shared memory layout, offsets from a 1024-aligned base
    static constexpr int kOffX = 0;
    static constexpr int kOffPk = kOffX + kStages * kXBytes;
    static constexpr int kOffSc = kOffPk + kStages * kChunkBytes;
    static constexpr int kOffBar = kOffSc + kStages * kScaleSlotBytes;
    // barriers: full[S], empty[S], afull[4], aempty[4], dfull[2], dempty[2], teardown
    static constexpr int kNumBars = 2 * kStages + 2 * kAStages + 4 + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 64 + 1024;  // + alignment slack
    static_assert(kXBytes % 1024 == 0, "X stages must stay 1024-byte aligned");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
    static_assert(kColsUsed <= 512, "tensor memory");
};

__device__ __forceinline__ long long cta_begin(const GemmParams& p, int c)
{
    return (long long)c * p.total_iters / p.grid;
}

// The CTA whose range holds iteration i.
__device__ __forceinline__ int cta_of(const GemmParams& p, long long i)
{
    int c = (int)((i * p.grid) / p.total_iters);
    while (c + 1 < p.grid && cta_begin(p, c + 1) <= i) ++c;
    while (c > 0 && cta_begin(p, c) > i) --c;
    return c;
}

// Partial slot of CTA c for tile t: 2c if t holds c's first iteration, else 2c+1.
__device__ __forceinline__ int slot_of(const GemmParams& p, int c, int t)
{
    return cta_begin(p, c) >= (long long)t * p.KC ? 2 * c : 2 * c + 1;
}

// Group range of chunk kc, clamped to the last group (chunks past K hold code 8).
__device__ __forceinline__ int group_lo(const GemmParams& p, int kc)
{
    return min(kc * kChunkK / p.G, p.ng - 1);
}

// (q - 8) * s as four FP16 pairs (k, k+1) ... (k+6, k+7) from one packed word whose
// nibble i holds k + 2*(i%4) + i/4: OR-ing a nibble into the mantissa of 1024.0
// gives 1024 + q (low nibble of a byte) or 1024 + 16q (high nibble), both exact.
__device__ __forceinline__ void dequant_word(uint32_t w, __half2 s2, uint32_t* out)
{
    const uint32_t lo = 0x000F000Fu, hi = 0x00F000F0u, magic = 0x64006400u;
    const __half2 c1032 = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
    const __half2 c1_16 = __halves2half2(__ushort_as_half(0x2C00), __ushort_as_half(0x2C00));
    const __half2 cm72 = __halves2half2(__ushort_as_half(0xD480), __ushort_as_half(0xD480));
    const uint32_t w8 = w >> 8;
    const uint32_t a = and_or(w, lo, magic);   // nibbles 0, 4 -> k+0, k+1
    const uint32_t b = and_or(w, hi, magic);   // nibbles 1, 5 -> k+2, k+3
    const uint32_t c = and_or(w8, lo, magic);  // nibbles 2, 6 -> k+4, k+5
    const uint32_t d = and_or(w8, hi, magic);  // nibbles 3, 7 -> k+6, k+7
    __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), c1032);
    __half2 hb = __hfma2(*reinterpret_cast<const __half2*>(&b), c1_16, cm72);
    __half2 hc = __hsub2(*reinterpret_cast<const __half2*>(&c), c1032);
    __half2 hd = __hfma2(*reinterpret_cast<const __half2*>(&d), c1_16, cm72);
    ha = __hmul2(ha, s2);
    hb = __hmul2(hb, s2);
    hc = __hmul2(hc, s2);
    hd = __hmul2(hd, s2);
    out[0] = *reinterpret_cast<uint32_t*>(&ha);
    out[1] = *reinterpret_cast<uint32_t*>(&hb);
    out[2] = *reinterpret_cast<uint32_t*>(&hc);
    out[3] = *reinterpret_cast<uint32_t*>(&hd);
}

template <int TM>
__global__ void __launch_bounds__(kThreads, 1)
    w4a16_tc_kernel(const __grid_constant__ CUtensorMap tmap_x, const GemmParams p)
{
    using C = TcCfg<TM>;
    constexpr int S = C::kStages;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte alignment for the 128-byte-swizzled X tiles.
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t* smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
    const uint32_t sbase = smem_addr(smem);

    const uint32_t bar0 = sbase + C::kOffBar;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
    auto afull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
    auto aempty_bar = [&](int a) { return bar0 + 8u * (2 * S + kAStages + a); };
    auto dfull_bar = [&](int d) { return bar0 + 8u * (2 * S + 2 * kAStages + d); };
    auto dempty_bar = [&](int d) { return bar0 + 8u * (2 * S + 2 * kAStages + 2 + d); };
    const uint32_t teardown_bar = bar0 + 8u * (2 * S + 2 * kAStages + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 8);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 16);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const WaitCtl ctl{abort_flag, p.status, p.wait_limit_ns};

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 8 + 1);  // 8 dequant warps + MMA commit
        }
        for (int a = 0; a < kAStages; ++a) {
            mbar_init(afull_bar(a), 8);
            mbar_init(aempty_bar(a), 1);
        }
        for (int d = 0; d < 2; ++d) {
            mbar_init(dfull_bar(d), 1);
            mbar_init(dempty_bar(d), 4);
        }
        mbar_init(teardown_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 12 && lane == 0) prefetch_tmap(&tmap_x);
    if (warp == 13) {
        tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const int cta = blockIdx.x;
    const long long it_begin = cta_begin(p, cta);
    const long long it_end = cta_begin(p, cta + 1);

    if (warp == 12) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            long long issued = 0;
            bool ok = true;
            for (long long i = it_begin; ok && i < it_end;) {
                const int t = (int)(i / p.KC);
                const int kb = (int)(i - (long long)t * p.KC);
                const int ke = (int)min((long long)p.KC, kb + (it_end - i));
                const int nt = t / p.m_tiles, mt = t - nt * p.m_tiles;
                for (int kc = kb; kc < ke; ++kc) {
                    if (!wait_one(empty_bar(s), ph ^ 1, ctl)) { ok = false; break; }
                    const int g0 = group_lo(p, kc);
                    const int g1 = min((kc * kChunkK + kChunkK - 1) / p.G, p.ng - 1);
                    const uint32_t sc_bytes = (uint32_t)(g1 - g0 + 1) * 256u;
                    mbar_arrive_expect_tx(full_bar(s), C::kXBytes + kChunkBytes + sc_bytes);
                    tma_load_2d(sbase + C::kOffX + s * C::kXBytes, &tmap_x, full_bar(s), kc * kChunkK, mt * TM);
                    bulk_load(sbase + C::kOffPk + s * kChunkBytes,
                              p.packed + ((size_t)nt * p.KC + kc) * kChunkWords, kChunkBytes, full_bar(s));
                    bulk_load(sbase + C::kOffSc + s * kScaleSlotBytes,
                              p.scales + ((size_t)nt * p.ng + g0) * kTileN, sc_bytes, full_bar(s));
                    ++issued;
                    if (++s == S) { s = 0; ph ^= 1; }
                }
                i += ke - kb;
            }
            // Wind down: let the last copies land before the CTA can exit.
            const long long inflight = issued < S ? issued : S;
            for (long long k = 1; k <= inflight; ++k) {
                int ss = s - (int)k;
                uint32_t pp = ph;
                if (ss < 0) { ss += S; pp ^= 1; }
                wait_drain(full_bar(ss), pp, 1000000000LL);
            }
        }
    } else if (warp == 13) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(128, TM);
            int s = 0, a = 0, d = 0;
            uint32_t ph = 0, aph = 0, dph = 0;
            bool ok = true;
            for (long long i = it_begin; ok && i < it_end;) {
                const int t = (int)(i / p.KC);
                const int kb = (int)(i - (long long)t * p.KC);
                const int ke = (int)min((long long)p.KC, kb + (it_end - i));
                if (!wait_one(dempty_bar(d), dph ^ 1, ctl)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + C::kDCol + d * TM;
                for (int kc = kb; kc < ke; ++kc) {
                    if (!wait_one(full_bar(s), ph, ctl) || !wait_one(afull_bar(a), aph, ctl)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t x_addr = sbase + C::kOffX + s * C::kXBytes;
#pragma unroll
                    for (int kk = 0; kk < kChunkK / 16; ++kk) {
                        mma_f16_ts(d_tmem, tmem + C::kACol + a * 32 + kk * 8, smem_desc_k_sw128(x_addr + kk * 32),
                                   idesc, (kc > kb || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(empty_bar(s));
                    mma_commit(aempty_bar(a));
                    if (++s == S) { s = 0; ph ^= 1; }
                    if (++a == kAStages) { a = 0; aph ^= 1; }
                }
                if (!ok) break;
                mma_commit(dfull_bar(d));
                if (++d == C::kDBufs) { d = 0; dph ^= 1; }
                i += ke - kb;
            }
            // Wind down: every MMA issued so far completes before TMEM is freed.
            mma_commit(teardown_bar);
            wait_drain(teardown_bar, 0, 1000000000LL);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ dequant
        const int quarter = warp & 3;            // TMEM lanes 32*quarter .. +31
        const int half = (warp - 4) >> 2;         // K values 32*half .. +31 of each chunk
        const int n_in = quarter * 32 + lane;
        int s = 0, a = 0;
        uint32_t ph = 0, aph = 0;
        bool ok = true;
        for (long long i = it_begin; ok && i < it_end;) {
            const int t = (int)(i / p.KC);
            const int kb = (int)(i - (long long)t * p.KC);
            const int ke = (int)min((long long)p.KC, kb + (it_end - i));
            for (int kc = kb; kc < ke; ++kc) {
                if (!wait_warp(full_bar(s), ph, ctl)) { ok = false; break; }
                const uint4 pk = *reinterpret_cast<const uint4*>(smem + C::kOffPk + s * kChunkBytes +
                                                                 (half * kTileN + n_in) * 16);
                const int g0 = group_lo(p, kc);
                const int g = min((kc * kChunkK + half * 32) / p.G, p.ng - 1);
                const __half sc = *reinterpret_cast<const __half*>(smem + C::kOffSc + s * kScaleSlotBytes +
                                                                   ((g - g0) * kTileN + n_in) * 2);
                const __half2 s2 = __halves2half2(sc, sc);
                uint32_t v[16];
                dequant_word(pk.x, s2, v + 0);
                dequant_word(pk.y, s2, v + 4);
                dequant_word(pk.z, s2, v + 8);
                dequant_word(pk.w, s2, v + 12);
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(s));
                if (!wait_warp(aempty_bar(a), aph ^ 1, ctl)) { ok = false; break; }
                tc_fence_after();
                tmem_st16(tmem + ((uint32_t)(quarter * 32) << 16) + C::kACol + a * 32 + half * 16, v);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(afull_bar(a));
                if (++s == S) { s = 0; ph ^= 1; }
                if (++a == kAStages) { a = 0; aph ^= 1; }
            }
            i += ke - kb;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        const int n_in = warp * 32 + lane;
        int d = 0;
        uint32_t dph = 0;
        for (long long i = it_begin; i < it_end;) {
            const int t = (int)(i / p.KC);
            const int kb = (int)(i - (long long)t * p.KC);
            const int ke = (int)min((long long)p.KC, kb + (it_end - i));
            const int nt = t / p.m_tiles, mt = t - nt * p.m_tiles;
            const int n = nt * kTileN + n_in;
            const int m0 = mt * TM;
            const int valid = min(TM, p.M - m0);
            const int chunks = (valid + 15) >> 4;
            const bool split = (kb != 0 || ke != p.KC);
            // All four epilogue warps leave together: they share named barriers.
            const bool ok = wait_warp(dfull_bar(d), dph, ctl);
            if (named_bar_or(1, 128, !ok)) break;
            tc_fence_after();
            const uint32_t d_tmem = tmem + ((uint32_t)(warp * 32) << 16) + C::kDCol + d * TM;
            float* part = p.partials + (size_t)slot_of(p, cta, t) * TM * kTileN + n_in;
            for (int c = 0; c < chunks; ++c) {
                uint32_t r[16];
                tmem_ld16(d_tmem + c * 16, r);
                if (!split) {
                    if (n < p.N) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const int m = m0 + c * 16 + e;
                            if (m < p.M) p.y[(size_t)m * p.N + n] = __float2half_rn(__uint_as_float(r[e]));
                        }
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < 16; ++e) part[(size_t)(c * 16 + e) * kTileN] = __uint_as_float(r[e]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dempty_bar(d));
            if (++d == C::kDBufs) { d = 0; dph ^= 1; }
            i += ke - kb;

            if (split) {
                // Deterministic split-K fix-up: the last contributor sums every
                // contributor's partial in CTA order.
                __threadfence();
                named_bar_sync(1, 128);
                const int c_lo = cta_of(p, (long long)t * p.KC);
                const int c_hi = cta_of(p, (long long)t * p.KC + p.KC - 1);
                if (threadIdx.x == 0) {
                    const int prev = atomicAdd(p.counters + c_lo, 1);
                    const int last = (prev == c_hi - c_lo);
                    if (last) p.counters[c_lo] = 0;
                    *last_flag = last;
                }
                named_bar_sync(1, 128);
                const int last = *last_flag;
                if (last) {
                    __threadfence();
                    for (int col = 0; col < valid; ++col) {
                        float acc = 0.f;
                        for (int cc = c_lo; cc <= c_hi; ++cc) {
                            const float* src = p.partials + (size_t)slot_of(p, cc, t) * TM * kTileN;
                            acc += __ldcg(src + (size_t)col * kTileN + n_in);
                        }
                        if (n < p.N) p.y[(size_t)(m0 + col) * p.N + n] = __float2half_rn(acc);
                    }
                }
                named_bar_sync(1, 128);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 13) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem, C::kTmemCols);
    }
}

template <int TM>
cudaError_t launch_tc(const CUtensorMap& tmap, const GemmParams& p, cudaStream_t stream);

template <int TM>
cudaError_t setup_tc();

}  // namespace w4a16
