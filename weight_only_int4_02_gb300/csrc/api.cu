// C ABI of libw4a16.so: argument checks, the per-shape plan (dispatch), the
// per-device workspace, the TMA descriptor of X, and the launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdlib>
#include <mutex>

#include "gemm_tc.cuh"
#include "decode.cuh"
#include "gemv.cuh"
#include "w4a16.h"

namespace w4a16 {
cudaError_t launch_pack(const uint8_t* codes, const uint16_t* scales, uint32_t* packed, uint16_t* scales_packed,
                        int K, int N, int KC, int n_tiles, int ng, int sms, cudaStream_t stream);
cudaError_t launch_pack_zeros(const uint8_t* zeros, uint8_t* zeros_packed, int N, int n_tiles, int ng, int sms,
                              cudaStream_t stream);
cudaError_t launch_pack_sp(const uint8_t* codes, const uint16_t* scales, uint8_t* packed, uint16_t* scales_packed,
                           int K, int N, int SC, int n_tiles, int ng, int sms, unsigned long long* violations,
                           cudaStream_t stream);
cudaError_t launch_pack_w8(const uint8_t* codes, const uint16_t* scales, uint8_t* packed, uint16_t* scales_packed,
                           int K, int N, int KC, int n_tiles, int ng, int sms, cudaStream_t stream);
}

namespace {

using namespace w4a16;

// Self-test of the bounded waits: one warp waits, with the GEMM kernels' own
// wait_warp, on phase 0 of an mbarrier that nothing arrives on; after limit_ns the
// wait gives up, sets the error word and the kernel returns.
__global__ void wait_selftest_kernel(int* status, long long limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    const WaitCtl ctl{&abort_flag, status, limit_ns};
    wait_warp(smem_addr(&bar), 0, ctl);
}

cudaError_t launch_wait_selftest(int* status, long long limit_ns, cudaStream_t stream)
{
    wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
    return cudaGetLastError();
}

thread_local int t_last_cuda_error = 0;

w4a16_status from_cuda(cudaError_t e)
{
    if (e == cudaSuccess) return W4A16_OK;
    t_last_cuda_error = (int)e;
    return W4A16_ERR_CUDA;
}

// Workspace layout (fixed, whatever the shape): error word at 0, split-K
// counters at 256 (one int per CTA, at most kMaxGrid), FP32 partials after.
constexpr size_t kCountersOff = 256;
constexpr int kMaxGrid = 1024;
constexpr size_t kPartialsOff = kCountersOff + 4 * kMaxGrid;
constexpr int kMaxTileM = 256;
constexpr int kMinItersPerCta = 4;
// Split cost model for fewer tiles than work units (make_plan), fitted (least
// squares) to per-launch times on GB300 of the 4096x4096, 4096x12288 and
// 11008x4096 layers at M = 1 ... 128 over every tile-aligned split:
// µs per stage whose weights were prefetched into the ring before X arrived
// (up to `ring` stages), per stage streamed after it, and the split-K fix-up per
// split tile and per valid row and extra contributor.
struct SplitCost {
    double ring, prefetched_us, streamed_us, fixup_us, fixup_row_us;
};
// The per-row fix-up costs are the fitted ones divided by the ratio of warps that now
// reduce a unit's last tile (the whole CTA, 15 or 23 warps, against the 4 epilogue warps).
constexpr SplitCost kSplit16 = {8, 0.15, 0.40, 1.4, 0.006};     // 16- and 32-row tiles, 16 KB stages
constexpr SplitCost kSplit64 = {0, 0.525, 0.525, 2.6, 0.008};   // 64-row tiles, 16 KB stages
constexpr SplitCost kSplit128 = {0, 0.375, 0.375, 2.9, 0.006};  // 128-row tiles, 8 KB stages
constexpr SplitCost kSplit256 = {0, 0.70, 0.70, 3.0, 0.0043};   // 256-row tiles, 8 KB stages (prefill)

struct DeviceState {
    bool ready = false;
    int sms = 0;
    void* ws = nullptr;
    size_t ws_bytes = 0;
    int* gemv_status = nullptr;   // device address of the error word of the kernels without a workspace
};

// Error word of the kernels that need no workspace (the CUDA-core kernel and the
// decode kernel) when the caller passes none: a timeout of a bounded wait sets bit 0.
__device__ int g_gemv_status;

constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
long long g_wait_limit_ns = 1000000000LL;
// Ablation knobs, read once from the environment: W4A16_SPLIT forces the number of
// parts every tile is cut into when there are fewer tiles than SMs (clamped to what
// the shape allows); W4A16_MIN_ITERS forces the fewest stages a CTA takes when
// there are more; W4A16_SPLIT_ALL=1 puts every tile in the split region then (stream-K
// over the whole space, with no whole tiles). 0 keeps the dispatcher's own choice.
int g_force_split = 0;
int g_force_min_iters = 0;
int g_force_split_all = 0;
int g_force_tm = 0;   // W4A16_TILE_M: rows of X per tile (16, 32, 64, 128 or 256) for the tensor-core kernel
int g_force_cb = 0;   // W4A16_DECODE_CB: columns per block (16, 32, 48, 64, 80 or 128) for the decode kernel

int ceil_div(int a, int b) { return (a + b - 1) / b; }

int norm_group(int K, int G) { return G == -1 ? K : G; }

bool valid_sizes(int K, int N, int G)
{
    if (K <= 0 || N <= 0 || (K % 8) != 0 || (N % 8) != 0) return false;
    return G == 32 || G == 64 || G == 128 || G == K;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// log2(G) for G a power of two; 30 (every k in group 0) otherwise, where G = K.
int group_shift(int G)
{
    if ((G & (G - 1)) != 0) return 30;
    int sh = 0;
    while ((1 << sh) < G) ++sh;
    return sh;
}

// The CUDA-core kernel (path 1) serves the 4-bit FP16 format (plain or with the
// fused epilogue) for up to this many rows of X when it is forced. The dispatcher
// does not pick it by itself: it is ALU-bound (about 3.5 instructions per weight at
// 55% issue) and measured slower than the decode kernel on every decode layer
// (4096 x 4096 at one row of X: 8.0 against 5.3 us per launch).
constexpr int kGemvMaxM = 4;
// The decode kernel (path 3) serves the 4-bit FP16 format (plain or with the fused
// epilogue) for up to sixteen rows of X when K is a multiple of 32; the dispatcher
// picks it by itself for up to eight, where it measured faster than the tensor-core
// kernel on every decode layer (4096 x 4096: 5.3 against 7.9 us; 18432 x 73728:
// 121 against 138 us). From nine rows on the second half of X doubles its MMAs and
// the tensor-core kernel wins on all but the smallest layers (decode_applies).
constexpr int kDecodeMaxM = 16;
constexpr int kDecodeAutoMaxM = 8;
// Forced path (0 = the dispatcher's choice, 1 = CUDA-core kernel, 2 = tensor-core
// kernel, 3 = decode kernel, each where it applies), for tests and ablations.
std::atomic<int> g_force_path{0};

struct Plan {
    int path;     // 1 = CUDA-core kernel (one to four rows of X), 2 = tcgen05 kernel, 3 = decode kernel
    int tm;       // rows of X per tile (MMA N)
    int ksub;     // sub-chunks per pipeline stage (64 values of k; 128 for 2:4 sparse codes)
    int xblocks;  // 64-wide blocks of X per stage (the X tensor map's box depth)
    int m_tiles, n_tiles, KC, ng, iters;
    long long total;
    int sk_tiles; // tiles of the split region (the first ones); the rest are whole tiles
    int grid;     // CTAs, one work unit each
    size_t ws_bytes;
    int gemv_mr;  // path 1: rows of X the kernel is built for (1, 2, 4)
    int gemv_cw;  // path 1: output columns per block (8, 16, 32)
    int gemv_blocks;
    int dec_mr;   // path 3: rows of X the kernel is built for (8, 16)
    int dec_cb;   // path 3: output columns per block (16, 32, 48, 64, 80, 128)
};

size_t ws_bytes_for(int grid, int tm) { return kPartialsOff + (size_t)2 * grid * tm * kTileN * sizeof(float); }

// fmt: the weight format (kFmt*); 8-bit codes run 128-value stages at every tile
// height (16 KB of codes a stage, as 256 values of 4-bit codes). Every CTA loads
// its own X tiles: no clusters, no multicast between CTAs.
Plan make_plan(int M, int N, int K, int G, int sms, int fmt = kFmtW4)
{
    Plan P;
    P.path = 2;
    P.tm = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
    if (g_force_tm == 16 || g_force_tm == 32 || g_force_tm == 64 || g_force_tm == 128 || g_force_tm == 256)
        P.tm = g_force_tm;
    if (fmt == kFmtW4Sp && P.tm > 128) P.tm = 128;   // sparse stages leave no room for 256-row X tiles
    P.m_tiles = ceil_div(M, P.tm);
    P.n_tiles = ceil_div(N, kTileN);
    P.ksub = (fmt == kFmtW8 || fmt == kFmtW4Sp) ? 2 : P.tm <= 64 ? 4 : 2;
    P.xblocks = fmt == kFmtW4Sp ? 4 : P.ksub;
    P.KC = ceil_div(ceil_div(K, kChunkK), kKPad) * kKPad;
    P.iters = P.KC / P.xblocks;
    P.ng = ceil_div(K, G);
    P.total = (long long)P.n_tiles * P.m_tiles * P.iters;
    long long units = sms < kMaxGrid ? sms : kMaxGrid;
    const long long work_tiles = (long long)P.n_tiles * P.m_tiles;
    if (work_tiles < units) {
        // Fewer tiles than work units (CTAs): every tile is cut into the
        // same number s of parts, so that unit boundaries fall on tile boundaries
        // and each split tile has exactly s contributors. s trades the stages a
        // unit runs against the split-K fix-up, whose last contributor reads every
        // other partial (costs measured on GB300, kSplit*).
        const SplitCost& sc = P.tm <= 32 ? kSplit16 : P.tm == 64 ? kSplit64 : P.tm == 128 ? kSplit128 : kSplit256;
        const int rows = P.m_tiles == 1 ? M : P.tm;
        const long long s_max = units / work_tiles;
        long long best_s = 1;
        double best = 0.0;
        for (long long s = 1; s <= s_max && s <= P.iters; ++s) {
            const double n = (double)((P.iters + s - 1) / s);   // stages of the longest unit
            const double prefetched = n < sc.ring ? n : sc.ring;
            const double cost = prefetched * sc.prefetched_us + (n - prefetched) * sc.streamed_us +
                                (s > 1 ? sc.fixup_us + sc.fixup_row_us * rows * (double)(s - 1) : 0.0);
            if (s == 1 || cost < best) {
                best = cost;
                best_s = s;
            }
        }
        if (g_force_split > 0) best_s = g_force_split < s_max ? (g_force_split < P.iters ? g_force_split : P.iters) : s_max;
        if (best_s < 1) best_s = 1;
        units = work_tiles * best_s;
        P.sk_tiles = (int)work_tiles;
    } else {
        // Stream-K over every SM, but a work unit takes at least kMinItersPerCta
        // stages, and with 32 or more rows of X at least a quarter (32 rows) or a
        // half (64 and up) of a tile's stages: the last contributor of a split
        // tile reads every other contributor's partial, which costs about one
        // round trip per 16 rows.
        int min_iters = P.tm >= 64 ? P.iters / 2 : P.tm == 32 ? P.iters / 4 : 0;
        if (min_iters < kMinItersPerCta) min_iters = kMinItersPerCta;
        if (g_force_min_iters > 0) min_iters = g_force_min_iters;
        const long long by_work = (P.total + min_iters - 1) / min_iters;
        if (units > by_work) units = by_work;
        if (units < 1) units = 1;
        // Whole waves of tiles go to the CTAs whole, round-robin; the tiles past the
        // last whole wave are the split region, cut into one stream-K range per CTA
        // and run first, so their partials and fix-ups overlap the whole tiles' MMAs
        // and every CTA ends on a whole tile. A split tile's last contributor reads
        // every other contributor's partial, one round trip per few rows, so the region
        // must not spread a few tiles over many CTAs: with fewer tiles than half the
        // CTAs it takes one whole wave more (about two contributors a tile; measured:
        // 20 tiles over 152 CTAs, 7.6 contributors each, ran the 4096x22016 layer at
        // M = 128 in 61 us against 27). That also gives every CTA's range a stage.
        // 2:4 sparse codes on 128-row tiles keep stream-K over every tile: they stage X
        // only two deep (64 KB stages), and whole tiles taken round-robin have every CTA
        // read the same X stage at once (18432x73728 at M = 128: 175 -> 194 us; at M = 16
        // the whole tiles measured faster, 109 -> 106 us).
        const long long rest = work_tiles % units;
        const long long sk = (rest > 0 && 2 * rest < units) ? rest + units : rest;
        P.sk_tiles = (g_force_split_all || (fmt == kFmtW4Sp && P.tm >= 128)) ? (int)work_tiles : (int)sk;
    }
    if (units < 1) units = 1;
    P.grid = (int)units;
    P.ws_bytes = ws_bytes_for(P.grid, P.tm);
    return P;
}

// Path 1 (CUDA-core kernel) for a shape: blocks of 32 columns when that gives at
// least one block per SM, else of 16, one CTA per block.
Plan make_gemv_plan(int M, int N, int K, int G, int sms)
{
    Plan P = {};
    P.path = 1;
    P.gemv_mr = M <= 1 ? 1 : M <= 2 ? 2 : 4;
    P.gemv_cw = ceil_div(N, 32) >= sms ? 32 : 16;
    P.gemv_blocks = ceil_div(N, P.gemv_cw);
    P.grid = P.gemv_blocks;
    P.n_tiles = ceil_div(N, kTileN);
    P.KC = ceil_div(ceil_div(K, kChunkK), kKPad) * kKPad;
    P.ng = ceil_div(K, G);
    P.ws_bytes = 0;   // no workspace: no partial sum leaves a CTA
    return P;
}

bool gemv_applies(int M, int fmt, int force)
{
    return fmt == kFmtW4 && M <= kGemvMaxM && force == 1;
}

// Columns per block of the decode kernel (path 3; one CTA per block). Two CTAs share
// an SM, and a launch chained behind another takes the slots as they free, so an SM
// ends up with two CTAs of it or none and the busiest SMs hold two blocks: with eight
// rows of X, the narrowest block that gives more CTAs than SMs and at most two per SM
// (one wave); else 128 where the layer has two 128-column blocks per SM, 64 where it
// has one 64-column block per SM, and 16 below. Measured on GB300 (launches of one
// shape chained, M = 1): 4096 x 12288 7.5 us with 48 against 8.3 with 64; 4096 x 22016
// 10.8 with 80 against 14.1 with 64 and 14.6 with 128; 18432 x 73728 115 with 128 or
// 64; N = 4096 fastest with 16.
int decode_block_cols(int N, int mr, int sms)
{
    if (g_force_cb == 16 || g_force_cb == 32 || g_force_cb == 64 || g_force_cb == 128 ||
        (mr == 8 && (g_force_cb == 48 || g_force_cb == 80)))
        return g_force_cb;
    if (mr == 8)
        for (int cb : {16, 32, 48, 64, 80, 128}) {
            const int ctas = ceil_div(N, cb);
            if (ctas > sms && ctas <= 2 * sms) return cb;
        }
    return ceil_div(N, 128) >= 2 * sms ? 128 : ceil_div(N, 64) >= sms ? 64 : 16;
}

Plan make_decode_plan(int M, int N, int K, int G, int sms)
{
    Plan P = {};
    P.path = 3;
    P.dec_mr = M <= 8 ? 8 : 16;
    P.dec_cb = decode_block_cols(N, P.dec_mr, sms);
    P.grid = ceil_div(N, P.dec_cb);
    P.n_tiles = ceil_div(N, kTileN);
    P.KC = ceil_div(ceil_div(K, kChunkK), kKPad) * kKPad;
    P.ng = ceil_div(K, G);
    P.ws_bytes = 0;   // no workspace: no partial sum leaves a CTA
    return P;
}

// The decode kernel takes up to eight rows of X by itself, and nine to sixteen on a
// layer of at most 4096 x 4096 with one 16-column block per SM or more: there the
// tensor-core kernel's split-K exchange outweighs the second pair of warp-level MMAs
// (16 x 4096 x 4096: 6.9 against 8.3 us per launch; the wider and deeper decode layers
// stay faster on the tensor-core kernel from nine rows on).
bool decode_applies(int M, int N, int K, int sms, int fmt, int force)
{
    if (fmt != kFmtW4 || M > kDecodeMaxM || K % 32 != 0) return false;
    if (force != 0) return force == 3;
    return M <= kDecodeAutoMaxM || (N <= 4096 && K <= 4096 && N >= 16 * sms);
}

// The plan of a shape on this device.
Plan device_plan(const DeviceState* st, int M, int N, int K, int G, int fmt)
{
    const int force = g_force_path.load();
    if (decode_applies(M, N, K, st->sms, fmt, force)) return make_decode_plan(M, N, K, G, st->sms);
    if (gemv_applies(M, fmt, force)) {
        Plan P = make_gemv_plan(M, N, K, G, st->sms);
        // persistent: no more CTAs than the SMs hold at once
        const long long slots = (long long)st->sms * gemv_resident_ctas(P.gemv_mr, P.gemv_cw, false);
        if (P.grid > slots) P.grid = (int)slots;
        return P;
    }
    return make_plan(M, N, K, G, st->sms, fmt);
}

// Shared-memory attributes of every variant of one tile shape (epilogue x weight format).
template <int TM, int KSUB>
cudaError_t setup_shape()
{
    cudaError_t e;
    if ((e = setup_tc<TM, KSUB, false, kFmtW4>()) != cudaSuccess ||
        (e = setup_tc<TM, KSUB, true, kFmtW4>()) != cudaSuccess ||
        (e = setup_tc<TM, KSUB, false, kFmtW4Zp>()) != cudaSuccess ||
        (e = setup_tc<TM, KSUB, true, kFmtW4Zp>()) != cudaSuccess ||
        (e = setup_tc<TM, KSUB, false, kFmtW4Bf16>()) != cudaSuccess ||
        (e = setup_tc<TM, KSUB, true, kFmtW4Bf16>()) != cudaSuccess ||
        (e = setup_tc<TM, 2, false, kFmtW8>()) != cudaSuccess || (e = setup_tc<TM, 2, true, kFmtW8>()) != cudaSuccess)
        return e;
    if constexpr (TM <= 128) {
        if ((e = setup_tc<TM, 2, false, kFmtW4Sp>()) != cudaSuccess ||
            (e = setup_tc<TM, 2, true, kFmtW4Sp>()) != cudaSuccess)
            return e;
    }
    return cudaSuccess;
}

template <int TM, int KSUB>
cudaError_t launch_shape(const CUtensorMap& map, const GemmParams& p, bool epi, int fmt, cudaStream_t stream)
{
    switch (fmt) {
        case kFmtW4Zp:
            return epi ? launch_tc<TM, KSUB, true, kFmtW4Zp>(map, p, stream)
                       : launch_tc<TM, KSUB, false, kFmtW4Zp>(map, p, stream);
        case kFmtW8:
            return epi ? launch_tc<TM, 2, true, kFmtW8>(map, p, stream)
                       : launch_tc<TM, 2, false, kFmtW8>(map, p, stream);
        case kFmtW4Bf16:
            return epi ? launch_tc<TM, KSUB, true, kFmtW4Bf16>(map, p, stream)
                       : launch_tc<TM, KSUB, false, kFmtW4Bf16>(map, p, stream);
        case kFmtW4Sp:
            if constexpr (TM <= 128)
                return epi ? launch_tc<TM, 2, true, kFmtW4Sp>(map, p, stream)
                           : launch_tc<TM, 2, false, kFmtW4Sp>(map, p, stream);
            else
                return cudaErrorInvalidValue;   // the plan never picks 256-row tiles for sparse codes
        default:
            return epi ? launch_tc<TM, KSUB, true, kFmtW4>(map, p, stream)
                       : launch_tc<TM, KSUB, false, kFmtW4>(map, p, stream);
    }
}

w4a16_status device_state(DeviceState** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return from_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return W4A16_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return from_cuda(e);
        if (major != 10 || minor != 3) return W4A16_ERR_UNSUPPORTED;  // built for sm_103a only
        if ((e = setup_gemv()) != cudaSuccess || (e = setup_decode()) != cudaSuccess) return from_cuda(e);
        void* gs = nullptr;
        if ((e = cudaGetSymbolAddress(&gs, g_gemv_status)) != cudaSuccess) return from_cuda(e);
        st.gemv_status = static_cast<int*>(gs);
        if ((e = setup_shape<16, 4>()) != cudaSuccess || (e = setup_shape<32, 4>()) != cudaSuccess ||
            (e = setup_shape<64, 4>()) != cudaSuccess || (e = setup_shape<128, 2>()) != cudaSuccess ||
            (e = setup_shape<256, 2>()) != cudaSuccess)
            return from_cuda(e);
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess) return from_cuda(e);
            if (q != cudaDriverEntryPointSuccess || !fn) return W4A16_ERR_UNSUPPORTED;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
            if (const char* s = std::getenv("W4A16_WAIT_LIMIT_NS")) g_wait_limit_ns = std::atoll(s);
            if (const char* s = std::getenv("W4A16_SPLIT")) g_force_split = std::atoi(s);
            if (const char* s = std::getenv("W4A16_MIN_ITERS")) g_force_min_iters = std::atoi(s);
            if (const char* s = std::getenv("W4A16_SPLIT_ALL")) g_force_split_all = std::atoi(s);
            if (const char* s = std::getenv("W4A16_TILE_M")) g_force_tm = std::atoi(s);
            if (const char* s = std::getenv("W4A16_DECODE_CB")) g_force_cb = std::atoi(s);
        }
        st.sms = sms;
        st.ready = true;
    }
    *out = &st;
    return W4A16_OK;
}

// The library's own workspace on the current device, sized for the largest plan.
w4a16_status own_workspace(DeviceState* st, void** ws, size_t* bytes)
{
    std::lock_guard<std::mutex> lock(g_mu);
    if (!st->ws) {
        const int grid = st->sms < kMaxGrid ? st->sms : kMaxGrid;
        const size_t need = ws_bytes_for(grid, kMaxTileM);
        void* p = nullptr;
        cudaError_t e = cudaMalloc(&p, need);
        if (e != cudaSuccess) return from_cuda(e);
        if ((e = cudaMemset(p, 0, need)) != cudaSuccess || (e = cudaDeviceSynchronize()) != cudaSuccess) {
            cudaFree(p);
            return from_cuda(e);
        }
        st->ws = p;
        st->ws_bytes = need;
    }
    *ws = st->ws;
    *bytes = st->ws_bytes;
    return W4A16_OK;
}

// X (rows ldx elements apart) as a 3-D view {64, M, K/64} (strides 2 ldx and 128
// bytes) when K is a multiple of 64, so one TMA brings a stage's KSUB blocks of 64
// columns; else the plain 2-D map {K, M}, one TMA per block, with the ragged K edge
// zero-filled.
bool encode_x_map(CUtensorMap* map, const void* x, int M, int K, int ldx, int rows, int ksub, bool allow_3d,
                  int* is_3d, bool bf16 = false)
{
    const CUtensorMapDataType dtype = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint32_t estr[3] = {1, 1, 1};
    if (allow_3d && K % kChunkK == 0) {
        cuuint64_t dims[3] = {(cuuint64_t)kChunkK, (cuuint64_t)M, (cuuint64_t)(K / kChunkK)};
        cuuint64_t strides[2] = {(cuuint64_t)ldx * 2, (cuuint64_t)kChunkK * 2};
        cuuint32_t box[3] = {(cuuint32_t)kChunkK, (cuuint32_t)rows, (cuuint32_t)ksub};
        CUresult r = g_encode(map, dtype, 3, const_cast<void*>(x), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r == CUDA_SUCCESS) {
            *is_3d = 1;
            return true;
        }
    }
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    cuuint64_t strides[1] = {(cuuint64_t)ldx * 2};
    cuuint32_t box[2] = {(cuuint32_t)kChunkK, (cuuint32_t)rows};
    CUresult r = g_encode(map, dtype, 2, const_cast<void*>(x), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    *is_3d = 0;
    return r == CUDA_SUCCESS;
}

// Tensor maps of the CUDA-core kernel: the packed words as uint32
// [n_tiles * tile_rows][512] (one row = 32 values of k for a tile's 128 columns),
// boxes of 32 rows x cb columns; the tile-ordered scales as 16-bit
// [n_tiles * ng][128], boxes of scale_rows groups x cb columns.
bool encode_gemv_maps(CUtensorMap* tw, CUtensorMap* ts, const void* packed, const void* scales, int n_tiles,
                      int tile_rows, int ng, int cb, int scale_rows)
{
    cuuint32_t estr[2] = {1, 1};
    cuuint64_t wdims[2] = {512, (cuuint64_t)n_tiles * tile_rows};
    cuuint64_t wstrides[1] = {2048};
    cuuint32_t wbox[2] = {(cuuint32_t)cb * 4, (cuuint32_t)(kGemvStageK / 32)};
    CUresult r = g_encode(tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(packed), wdims, wstrides, wbox,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    cuuint64_t sdims[2] = {128, (cuuint64_t)n_tiles * ng};
    cuuint64_t sstrides[1] = {256};
    cuuint32_t sbox[2] = {(cuuint32_t)cb, (cuuint32_t)scale_rows};
    r = g_encode(ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(scales), sdims, sstrides, sbox, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor maps of the decode kernel: the packed words as uint32 [n_tiles * tile_rows][512],
// boxes of 16 rows x cb columns; the tile-ordered scales as 16-bit [n_tiles * ng][128],
// boxes of scale_rows groups x cb columns; X as the 3-D view {32, M, K/32} (strides
// 2 ldx and 64 bytes; K is a multiple of 32), boxes of 32 values x M rows x 16 (every
// box in bounds: out-of-bounds rows measured slow to fill).
bool encode_decode_maps(CUtensorMap* tw, CUtensorMap* ts, CUtensorMap* tx, const void* packed, const void* scales,
                        const void* x, int n_tiles, int tile_rows, int ng, int cb, int scale_rows, int M, int K,
                        int ldx)
{
    cuuint32_t estr[3] = {1, 1, 1};
    cuuint64_t wdims[2] = {512, (cuuint64_t)n_tiles * tile_rows};
    cuuint64_t wstrides[1] = {2048};
    // boxes of up to 64 columns (128: two boxes); 48 and 80 columns: boxes of 16
    const bool narrow = cb == 48 || cb == 80;
    const int box_cols = narrow ? 16 : cb < 64 ? cb : 64;
    cuuint32_t wbox[2] = {(cuuint32_t)box_cols * 4, (cuuint32_t)kDecStageRows};
    CUresult r = g_encode(tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(packed), wdims, wstrides, wbox,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    cuuint64_t sdims[2] = {128, (cuuint64_t)n_tiles * ng};
    cuuint64_t sstrides[1] = {256};
    cuuint32_t sbox[2] = {(cuuint32_t)(narrow ? 16 : cb), (cuuint32_t)scale_rows};
    r = g_encode(ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(scales), sdims, sstrides, sbox, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    cuuint64_t xdims[3] = {32, (cuuint64_t)M, (cuuint64_t)(K / 32)};
    cuuint64_t xstrides[2] = {(cuuint64_t)ldx * 2, 64};
    cuuint32_t xbox[3] = {32, (cuuint32_t)M, (cuuint32_t)kDecStageRows};
    r = g_encode(tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(x), xdims, xstrides, xbox, estr,
                 CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

w4a16_status gemm_impl(const uint16_t* x, const uint32_t* packed, const uint16_t* scales_packed, uint16_t* y, int M,
                       int N, int K, int G, void* ws, size_t ws_bytes, bool own_ws, cudaStream_t stream,
                       const uint16_t* bias = nullptr, const uint16_t* residual = nullptr, int act = 0,
                       int fmt = kFmtW4, const uint8_t* zeros_packed = nullptr, int ldx = 0, int ldy = 0,
                       int ldr = 0)
{
    if ((fmt == kFmtW4Zp) != (zeros_packed != nullptr)) return W4A16_ERR_INVALID_ARG;
    G = norm_group(K, G);
    if (M < 0 || !valid_sizes(K, N, G)) return W4A16_ERR_INVALID_ARG;
    // Row strides in elements (0: the dense [M][K] and [M][N] layouts). X rows start on
    // 16-byte boundaries (the TMA maps' strides): ldx is a multiple of 8.
    if (ldx == 0) ldx = K;
    if (ldy == 0) ldy = N;
    if (ldr == 0) ldr = N;
    if (ldx < K || ldx % 8 != 0 || ldy < N || ldr < N) return W4A16_ERR_INVALID_ARG;
    if (M == 0) return W4A16_OK;
    if (!x || !packed || !scales_packed || !y) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(packed) || !aligned16(scales_packed) || !aligned16(y) ||
        (zeros_packed && !aligned16(zeros_packed)))
        return W4A16_ERR_INVALID_ARG;
    if (!own_ws && (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) != 0)) return W4A16_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    w4a16_status rc = device_state(&st);
    if (rc != W4A16_OK) return rc;
    const Plan P = device_plan(st, M, N, K, G, fmt);
    // the tensor-core kernel counts a CTA's stages in 32 bits
    if (P.path == 2 && P.total >= (1LL << 31)) return W4A16_ERR_INVALID_ARG;
    if (P.path == 3) {
        DecodeParams d;
        d.y = reinterpret_cast<__half*>(y);
        d.bias = reinterpret_cast<const __half*>(bias);
        d.residual = reinterpret_cast<const __half*>(residual);
        d.ldy = ldy;
        d.ldr = ldr;
        // a timeout is reported in the caller's workspace (or the no-allocation
        // array) when one is given, else in the library's own word for these kernels
        d.status = own_ws ? st->gemv_status : reinterpret_cast<int*>(ws);
        d.wait_limit_ns = g_wait_limit_ns;
        d.act = act;
        d.M = M;
        d.N = N;
        d.ng = P.ng;
        d.g_shift = group_shift(G);
        d.tile_rows = 2 * P.KC;
        d.rows = K / 32;
        d.stages = ceil_div(d.rows, kDecStageRows);
        d.scale_rows = ((G & (G - 1)) == 0 && G <= kDecStageRows * 32) ? kDecStageRows * 32 / G : 1;
        d.x_rows = M;
        // slots for 24 to 80 KB of packed words in flight (decode_words_in_flight), within
        // the shared-memory budget
        d.ring = decode_words_in_flight(P.dec_cb) / (kDecStageRows * P.dec_cb * 16);
        if (d.ring > kDecSmemBudget / decode_slot_bytes(P.dec_cb, M)) d.ring = kDecSmemBudget / decode_slot_bytes(P.dec_cb, M);
        if (d.ring > kDecMaxRing) d.ring = kDecMaxRing;
        if (d.ring < 2) return W4A16_ERR_INVALID_ARG;   // cannot happen for M <= 16
        CUtensorMap tw, ts, tx;
        if (!encode_decode_maps(&tw, &ts, &tx, packed, scales_packed, x, P.n_tiles, d.tile_rows, P.ng, P.dec_cb,
                                d.scale_rows, M, K, ldx))
            return W4A16_ERR_INVALID_ARG;
        const bool epi = bias || residual || act != 0;
        return from_cuda(launch_decode(tw, ts, tx, d, P.dec_mr, P.dec_cb, epi, P.grid, stream));
    }
    if (P.path == 1) {
        GemvParams g;
        g.x = reinterpret_cast<const __half*>(x);
        g.y = reinterpret_cast<__half*>(y);
        g.ldx = ldx;
        g.ldy = ldy;
        g.ldr = ldr;
        g.bias = reinterpret_cast<const __half*>(bias);
        g.residual = reinterpret_cast<const __half*>(residual);
        // a timeout is reported in the caller's workspace (or the no-allocation
        // array) when one is given, else in the library's own word for this kernel
        g.status = own_ws ? st->gemv_status : reinterpret_cast<int*>(ws);
        g.wait_limit_ns = g_wait_limit_ns;
        g.act = act;
        g.M = M;
        g.N = N;
        g.K = K;
        g.ng = P.ng;
        g.g_shift = group_shift(G);
        g.tile_rows = 2 * P.KC;
        g.rows = ceil_div(K, 32);
        g.stages = ceil_div(g.rows, kGemvStageK / 32);
        g.scale_rows = ((G & (G - 1)) == 0 && G <= kGemvStageK) ? kGemvStageK / G : 1;
        g.blocks = P.gemv_blocks;
        CUtensorMap tw, ts;
        if (!encode_gemv_maps(&tw, &ts, packed, scales_packed, P.n_tiles, g.tile_rows, P.ng, P.gemv_cw, g.scale_rows))
            return W4A16_ERR_INVALID_ARG;
        const bool epi = bias || residual || act != 0;
        // persistent: no more CTAs than the SMs hold at once; CTAs take blocks in turn
        const long long slots = (long long)st->sms * gemv_resident_ctas(P.gemv_mr, P.gemv_cw, epi);
        const int grid = (int)(P.gemv_blocks < slots ? P.gemv_blocks : slots);
        return from_cuda(launch_gemv(tw, ts, g, P.gemv_mr, P.gemv_cw, epi, grid, stream));
    }
    if (own_ws) {
        rc = own_workspace(st, &ws, &ws_bytes);
        if (rc != W4A16_OK) return rc;
    }
    if (ws_bytes < P.ws_bytes) return W4A16_ERR_WORKSPACE;

    GemmParams p;
    p.packed = packed;
    p.scales = reinterpret_cast<const __half*>(scales_packed);
    p.zeros = zeros_packed;
    p.y = reinterpret_cast<__half*>(y);
    p.status = reinterpret_cast<int*>(ws);
    p.counters = reinterpret_cast<int*>(static_cast<char*>(ws) + kCountersOff);
    p.partials = reinterpret_cast<float*>(static_cast<char*>(ws) + kPartialsOff);
    p.M = M;
    p.N = N;
    p.K = K;
    p.G = G;
    p.ng = P.ng;
    p.g_shift = group_shift(G);
    p.n_tiles = P.n_tiles;
    p.m_tiles = P.m_tiles;
    p.KC = fmt == kFmtW4Sp ? P.KC / 2 : P.KC;   // packed chunks per column (128 values of k when sparse)
    p.iters = P.iters;
    p.sk_tiles = P.sk_tiles;
    p.sk_iters = (long long)P.sk_tiles * P.iters;
    p.grid = P.grid;
    p.wait_limit_ns = g_wait_limit_ns;
    p.bias = reinterpret_cast<const __half*>(bias);
    p.residual = reinterpret_cast<const __half*>(residual);
    p.act = act;
    p.ldy = ldy;
    p.ldr = ldr;

    CUtensorMap map;
    // With one row tile, a box of M rows rounded up to the 8-row swizzle atom is
    // enough: MMA rows past M feed only output columns that are never stored.
    p.x_rows = P.m_tiles == 1 ? ((M + 7) / 8) * 8 : P.tm;
    if (!encode_x_map(&map, x, M, K, ldx, p.x_rows, P.xblocks, true, &p.x_3d, fmt == kFmtW4Bf16))
        return W4A16_ERR_INVALID_ARG;
    cudaError_t e;
    const bool epi = bias || residual || act != 0;
    switch (P.tm) {
        case 16: e = launch_shape<16, 4>(map, p, epi, fmt, stream); break;
        case 32: e = launch_shape<32, 4>(map, p, epi, fmt, stream); break;
        case 64: e = launch_shape<64, 4>(map, p, epi, fmt, stream); break;
        case 128: e = launch_shape<128, 2>(map, p, epi, fmt, stream); break;
        default: e = launch_shape<256, 2>(map, p, epi, fmt, stream); break;
    }
    return from_cuda(e);
}

// The no-allocation array's device address on the current device, or null if no
// no-allocation call has looked it up yet (defined with that entry point below).
void* noalloc_scratch_if_set();

}  // namespace

extern "C" {

int w4a16_layout_version(void) { return 2; }

const char* w4a16_status_string(int status)
{
    switch (status) {
        case W4A16_OK: return "ok";
        case W4A16_ERR_INVALID_ARG: return "invalid argument";
        case W4A16_ERR_UNSUPPORTED: return "unsupported device";
        case W4A16_ERR_CUDA: return "CUDA error";
        case W4A16_ERR_TIMEOUT: return "a kernel wait timed out";
        case W4A16_ERR_WORKSPACE: return "workspace too small";
        default: return "unknown status";
    }
}

int w4a16_last_cuda_error(void) { return t_last_cuda_error; }

size_t w4a16_packed_words(int K, int N, int group_size)
{
    if (!valid_sizes(K, N, norm_group(K, group_size))) return 0;
    return (size_t)ceil_div(N, kTileN) * (ceil_div(ceil_div(K, kChunkK), kKPad) * kKPad) * kChunkWords;
}

size_t w4a16_scales_elems(int K, int N, int group_size)
{
    const int G = norm_group(K, group_size);
    if (!valid_sizes(K, N, G)) return 0;
    return (size_t)ceil_div(N, kTileN) * ceil_div(K, G) * kTileN;
}

w4a16_status w4a16_pack(const uint8_t* codes, const uint16_t* scales, uint32_t* packed, uint16_t* scales_packed,
                        int K, int N, int group_size, w4a16_stream_t stream)
{
    const int G = norm_group(K, group_size);
    if (!valid_sizes(K, N, G)) return W4A16_ERR_INVALID_ARG;
    if (!codes || !scales || !packed || !scales_packed) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(packed) || !aligned16(scales_packed)) return W4A16_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    w4a16_status rc = device_state(&st);
    if (rc != W4A16_OK) return rc;
    return from_cuda(launch_pack(codes, scales, packed, scales_packed, K, N,
                                 ceil_div(ceil_div(K, kChunkK), kKPad) * kKPad,
                                 ceil_div(N, kTileN), ceil_div(K, G), st->sms,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_gemm(const uint16_t* x, const uint32_t* packed, const uint16_t* scales_packed, uint16_t* y, int M,
                        int N, int K, int group_size, w4a16_stream_t stream)
{
    return gemm_impl(x, packed, scales_packed, y, M, N, K, group_size, nullptr, 0, true,
                     reinterpret_cast<cudaStream_t>(stream));
}

size_t w4a16_workspace_bytes(int M, int N, int K, int group_size)
{
    const int G = norm_group(K, group_size);
    if (M < 0 || !valid_sizes(K, N, G)) return 0;
    DeviceState* st = nullptr;
    int sms = kMaxGrid;
    if (device_state(&st) == W4A16_OK) sms = st->sms;
    if (M == 0) return kPartialsOff;
    // enough for every weight format's plan
    size_t need = 0;
    for (int fmt : {kFmtW4, kFmtW8, kFmtW4Sp}) {
        const size_t b = make_plan(M, N, K, G, sms, fmt).ws_bytes;
        need = b > need ? b : need;
    }
    return need;
}

w4a16_status w4a16_gemm_ws(const uint16_t* x, const uint32_t* packed, const uint16_t* scales_packed, uint16_t* y,
                           int M, int N, int K, int group_size, void* workspace, size_t ws_bytes,
                           w4a16_stream_t stream)
{
    return gemm_impl(x, packed, scales_packed, y, M, N, K, group_size, workspace, ws_bytes, false,
                     reinterpret_cast<cudaStream_t>(stream));
}

w4a16_status w4a16_gemm_fused(const uint16_t* x, const uint32_t* packed, const uint16_t* scales_packed,
                              uint16_t* y, int M, int N, int K, int group_size, const uint16_t* bias,
                              const uint16_t* residual, int activation, void* workspace, size_t ws_bytes,
                              w4a16_stream_t stream)
{
    if (activation < W4A16_ACT_NONE || activation > W4A16_ACT_RELU) return W4A16_ERR_INVALID_ARG;
    if ((bias && (reinterpret_cast<uintptr_t>(bias) & 1)) || (residual && (reinterpret_cast<uintptr_t>(residual) & 1)))
        return W4A16_ERR_INVALID_ARG;
    return gemm_impl(x, packed, scales_packed, y, M, N, K, group_size, workspace, ws_bytes, workspace == nullptr,
                     reinterpret_cast<cudaStream_t>(stream), bias, residual, activation);
}

w4a16_status w4a16_gemm_strided(const uint16_t* x, int ldx, const uint32_t* packed, const uint16_t* scales_packed,
                                uint16_t* y, int ldy, int M, int N, int K, int group_size, const uint16_t* bias,
                                const uint16_t* residual, int ldr, int activation, void* workspace, size_t ws_bytes,
                                w4a16_stream_t stream)
{
    if (activation < W4A16_ACT_NONE || activation > W4A16_ACT_RELU) return W4A16_ERR_INVALID_ARG;
    if ((bias && (reinterpret_cast<uintptr_t>(bias) & 1)) || (residual && (reinterpret_cast<uintptr_t>(residual) & 1)))
        return W4A16_ERR_INVALID_ARG;
    if (ldx <= 0 || ldy <= 0 || (residual && ldr <= 0)) return W4A16_ERR_INVALID_ARG;
    return gemm_impl(x, packed, scales_packed, y, M, N, K, group_size, workspace, ws_bytes, workspace == nullptr,
                     reinterpret_cast<cudaStream_t>(stream), bias, residual, activation, kFmtW4, nullptr, ldx, ldy,
                     residual ? ldr : N);
}

size_t w4a16_zeros_bytes(int K, int N, int group_size)
{
    const int G = norm_group(K, group_size);
    if (!valid_sizes(K, N, G)) return 0;
    return (size_t)ceil_div(N, kTileN) * ceil_div(K, G) * (kTileN / 2);
}

w4a16_status w4a16_pack_zeros(const uint8_t* zeros, uint8_t* zeros_packed, int K, int N, int group_size,
                              w4a16_stream_t stream)
{
    const int G = norm_group(K, group_size);
    if (!valid_sizes(K, N, G)) return W4A16_ERR_INVALID_ARG;
    if (!zeros || !zeros_packed || !aligned16(zeros_packed)) return W4A16_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    w4a16_status rc = device_state(&st);
    if (rc != W4A16_OK) return rc;
    return from_cuda(launch_pack_zeros(zeros, zeros_packed, N, ceil_div(N, kTileN), ceil_div(K, G), st->sms,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_gemm_zp(const uint16_t* x, const uint32_t* packed, const uint16_t* scales_packed,
                           const uint8_t* zeros_packed, uint16_t* y, int M, int N, int K, int group_size,
                           const uint16_t* bias, const uint16_t* residual, int activation, void* workspace,
                           size_t ws_bytes, w4a16_stream_t stream)
{
    if (!zeros_packed && M != 0) return W4A16_ERR_INVALID_ARG;
    if (activation < W4A16_ACT_NONE || activation > W4A16_ACT_RELU) return W4A16_ERR_INVALID_ARG;
    if ((bias && (reinterpret_cast<uintptr_t>(bias) & 1)) || (residual && (reinterpret_cast<uintptr_t>(residual) & 1)))
        return W4A16_ERR_INVALID_ARG;
    return gemm_impl(x, packed, scales_packed, y, M, N, K, group_size, workspace, ws_bytes, workspace == nullptr,
                     reinterpret_cast<cudaStream_t>(stream), bias, residual, activation, kFmtW4Zp, zeros_packed);
}

w4a16_status w4a16_bf16_gemm(const uint16_t* x, const uint32_t* packed, const uint16_t* scales_packed, uint16_t* y,
                             int M, int N, int K, int group_size, const uint16_t* bias, const uint16_t* residual,
                             int activation, void* workspace, size_t ws_bytes, w4a16_stream_t stream)
{
    if (activation < W4A16_ACT_NONE || activation > W4A16_ACT_RELU) return W4A16_ERR_INVALID_ARG;
    if ((bias && (reinterpret_cast<uintptr_t>(bias) & 1)) || (residual && (reinterpret_cast<uintptr_t>(residual) & 1)))
        return W4A16_ERR_INVALID_ARG;
    return gemm_impl(x, packed, scales_packed, y, M, N, K, group_size, workspace, ws_bytes, workspace == nullptr,
                     reinterpret_cast<cudaStream_t>(stream), bias, residual, activation, kFmtW4Bf16);
}

size_t w4a16_sp_packed_bytes(int K, int N, int group_size)
{
    if (!valid_sizes(K, N, norm_group(K, group_size))) return 0;
    return (size_t)ceil_div(N, kTileN) * (ceil_div(ceil_div(K, kChunkK), kKPad) * kKPad / 2) * (kChunkBytes + 2048);
}

w4a16_status w4a16_sp_pack(const uint8_t* codes, const uint16_t* scales, uint8_t* packed, uint16_t* scales_packed,
                           int K, int N, int group_size, unsigned long long* violations, w4a16_stream_t stream)
{
    const int G = norm_group(K, group_size);
    if (!valid_sizes(K, N, G)) return W4A16_ERR_INVALID_ARG;
    if (!codes || !scales || !packed || !scales_packed) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(packed) || !aligned16(scales_packed) || (reinterpret_cast<uintptr_t>(violations) & 7))
        return W4A16_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    w4a16_status rc = device_state(&st);
    if (rc != W4A16_OK) return rc;
    return from_cuda(launch_pack_sp(codes, scales, packed, scales_packed, K, N,
                                    ceil_div(ceil_div(K, kChunkK), kKPad) * kKPad / 2, ceil_div(N, kTileN),
                                    ceil_div(K, G), st->sms, violations, reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_sp_gemm(const uint16_t* x, const uint8_t* packed, const uint16_t* scales_packed, uint16_t* y,
                           int M, int N, int K, int group_size, const uint16_t* bias, const uint16_t* residual,
                           int activation, void* workspace, size_t ws_bytes, w4a16_stream_t stream)
{
    if (activation < W4A16_ACT_NONE || activation > W4A16_ACT_RELU) return W4A16_ERR_INVALID_ARG;
    if ((bias && (reinterpret_cast<uintptr_t>(bias) & 1)) || (residual && (reinterpret_cast<uintptr_t>(residual) & 1)))
        return W4A16_ERR_INVALID_ARG;
    return gemm_impl(x, reinterpret_cast<const uint32_t*>(packed), scales_packed, y, M, N, K, group_size, workspace,
                     ws_bytes, workspace == nullptr, reinterpret_cast<cudaStream_t>(stream), bias, residual,
                     activation, kFmtW4Sp);
}

size_t w4a16_w8_packed_bytes(int K, int N, int group_size)
{
    if (!valid_sizes(K, N, norm_group(K, group_size))) return 0;
    return (size_t)ceil_div(N, kTileN) * (ceil_div(ceil_div(K, kChunkK), kKPad) * kKPad) * (2 * kChunkBytes);
}

w4a16_status w4a16_w8_pack(const uint8_t* codes, const uint16_t* scales, uint8_t* packed, uint16_t* scales_packed,
                           int K, int N, int group_size, w4a16_stream_t stream)
{
    const int G = norm_group(K, group_size);
    if (!valid_sizes(K, N, G)) return W4A16_ERR_INVALID_ARG;
    if (!codes || !scales || !packed || !scales_packed) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(packed) || !aligned16(scales_packed)) return W4A16_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    w4a16_status rc = device_state(&st);
    if (rc != W4A16_OK) return rc;
    return from_cuda(launch_pack_w8(codes, scales, packed, scales_packed, K, N,
                                    ceil_div(ceil_div(K, kChunkK), kKPad) * kKPad, ceil_div(N, kTileN),
                                    ceil_div(K, G), st->sms, reinterpret_cast<cudaStream_t>(stream)));
}

w4a16_status w4a16_w8_gemm(const uint16_t* x, const uint8_t* packed, const uint16_t* scales_packed, uint16_t* y,
                           int M, int N, int K, int group_size, const uint16_t* bias, const uint16_t* residual,
                           int activation, void* workspace, size_t ws_bytes, w4a16_stream_t stream)
{
    if (activation < W4A16_ACT_NONE || activation > W4A16_ACT_RELU) return W4A16_ERR_INVALID_ARG;
    if ((bias && (reinterpret_cast<uintptr_t>(bias) & 1)) || (residual && (reinterpret_cast<uintptr_t>(residual) & 1)))
        return W4A16_ERR_INVALID_ARG;
    return gemm_impl(x, reinterpret_cast<const uint32_t*>(packed), scales_packed, y, M, N, K, group_size, workspace,
                     ws_bytes, workspace == nullptr, reinterpret_cast<cudaStream_t>(stream), bias, residual,
                     activation, kFmtW8);
}

w4a16_status w4a16_selftest_wait_timeout(void* workspace, long long limit_ns, w4a16_stream_t stream)
{
    if (limit_ns <= 0 || limit_ns > 10000000000LL) return W4A16_ERR_INVALID_ARG;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return W4A16_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    w4a16_status rc = device_state(&st);
    if (rc != W4A16_OK) return rc;
    if (!workspace) {
        size_t bytes = 0;
        if ((rc = own_workspace(st, &workspace, &bytes)) != W4A16_OK) return rc;
    }
    return from_cuda(launch_wait_selftest(reinterpret_cast<int*>(workspace), limit_ns,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

// Reads the error word at the start of a workspace (or of the no-allocation
// array); after a timeout clears the word and the split-K counters.
w4a16_status read_and_clear_status(void* ws, bool* timed_out)
{
    int word = 0;
    cudaError_t e = cudaMemcpy(&word, ws, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return from_cuda(e);
    if (word == 0) return W4A16_OK;
    *timed_out = true;
    if ((e = cudaMemset(ws, 0, kPartialsOff)) != cudaSuccess || (e = cudaDeviceSynchronize()) != cudaSuccess)
        return from_cuda(e);
    return W4A16_OK;
}

// Reads and clears one error word (no counters beside it).
w4a16_status read_and_clear_word(int* word_dev, bool* timed_out)
{
    int word = 0;
    cudaError_t e = cudaMemcpy(&word, word_dev, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return from_cuda(e);
    if (word == 0) return W4A16_OK;
    *timed_out = true;
    if ((e = cudaMemset(word_dev, 0, sizeof(int))) != cudaSuccess || (e = cudaDeviceSynchronize()) != cudaSuccess)
        return from_cuda(e);
    return W4A16_OK;
}

w4a16_status w4a16_check_device_status(void* workspace, w4a16_stream_t stream)
{
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return from_cuda(e);
    bool timed_out = false;
    w4a16_status rc = W4A16_OK;
    if (workspace) {
        rc = read_and_clear_status(workspace, &timed_out);
    } else {
        DeviceState* st = nullptr;
        if ((rc = device_state(&st)) != W4A16_OK) return rc;
        // the library's own workspace, the CUDA-core kernel's word, and the
        // no-allocation array once it is in use
        if (st->ws) rc = read_and_clear_status(st->ws, &timed_out);
        if (rc == W4A16_OK) rc = read_and_clear_word(st->gemv_status, &timed_out);
        void* na = noalloc_scratch_if_set();
        if (rc == W4A16_OK && na) rc = read_and_clear_status(na, &timed_out);
    }
    if (rc != W4A16_OK) return rc;
    return timed_out ? W4A16_ERR_TIMEOUT : W4A16_OK;
}

w4a16_status w4a16_plan(int M, int N, int K, int group_size, int* path, int* tile_m, int* grid)
{
    const int G = norm_group(K, group_size);
    if (M <= 0 || !valid_sizes(K, N, G) || !path || !tile_m || !grid) return W4A16_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    w4a16_status rc = device_state(&st);
    if (rc != W4A16_OK) return rc;
    const Plan P = device_plan(st, M, N, K, G, kFmtW4);
    *path = P.path;
    *tile_m = P.path == 1 ? P.gemv_mr : P.path == 3 ? P.dec_mr : P.tm;
    *grid = P.grid;
    return W4A16_OK;
}

long long w4a16_set_wait_limit_ns(long long limit_ns)
{
    DeviceState* st = nullptr;
    device_state(&st);   // the first device set-up reads W4A16_WAIT_LIMIT_NS; set after it
    std::lock_guard<std::mutex> lock(g_mu);
    const long long prev = g_wait_limit_ns;
    if (limit_ns > 0) g_wait_limit_ns = limit_ns;
    return prev;
}

int w4a16_force_path(int path)
{
    if (path < 0 || path > 3) return -1;
    return g_force_path.exchange(path);
}


}  // extern "C"

// ------------------------------------------------------------------ no-allocation variant
// Some callers may not allocate device memory: plug-ins whose host framework owns
// every byte of GPU memory and hands out none, or latency-critical loops that
// cannot afford cudaMalloc's implicit device-wide synchronisation. For them,
// w4a16_gemm_noalloc runs the same GEMM with its split-K scratch (error word,
// tile counters, FP32 partials) in this fixed device array instead of a
// workspace. Every GPU that loads the library holds the array until exit.
namespace {

constexpr size_t kNoAllocBytes = (size_t)8 << 20;  // 8 MiB, W4A16_NOALLOC_MAX_BYTES
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per device.
w4a16_status noalloc_scratch(void** out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return from_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return W4A16_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return from_cuda(e);
        g_noalloc_ptr[dev] = ptr;
    }
    *out = g_noalloc_ptr[dev];
    return W4A16_OK;
}

void* noalloc_scratch_if_set()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    return g_noalloc_ptr[dev];
}

}  // namespace

extern "C" w4a16_status w4a16_gemm_noalloc(const uint16_t* x, const uint32_t* packed,
                                           const uint16_t* scales_packed, uint16_t* y, int M, int N, int K,
                                           int group_size, w4a16_stream_t stream)
{
    const int G = norm_group(K, group_size);
    if (M < 0 || !valid_sizes(K, N, G)) return W4A16_ERR_INVALID_ARG;
    if (M == 0) return W4A16_OK;
    // Every check that can refuse the call comes before anything is enqueued.
    if (!x || !packed || !scales_packed || !y) return W4A16_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(packed) || !aligned16(scales_packed) || !aligned16(y))
        return W4A16_ERR_INVALID_ARG;
    DeviceState* st = nullptr;
    w4a16_status rc = device_state(&st);
    if (rc != W4A16_OK) return rc;
    const Plan P = device_plan(st, M, N, K, G, kFmtW4);
    if (P.ws_bytes > kNoAllocBytes) return W4A16_ERR_WORKSPACE;
    void* scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc != W4A16_OK) return rc;
    if (P.path == 2) {
        // The split-K counters must start at zero; the array keeps whatever the
        // previous call left there. The error word (bytes 0..3) is left alone: it
        // holds a timeout until w4a16_check_device_status(NULL) reads and clears it.
        cudaError_t e = cudaMemsetAsync(static_cast<char*>(scratch) + kCountersOff, 0, kPartialsOff - kCountersOff,
                                        reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return from_cuda(e);
    }
    return gemm_impl(x, packed, scales_packed, y, M, N, K, G, scratch, kNoAllocBytes, false,
                     reinterpret_cast<cudaStream_t>(stream));
}

