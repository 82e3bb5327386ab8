// C ABI of libw4a16.so: argument checks, the per-shape plan (dispatch), the
// per-device workspace, the TMA descriptor of X, and the launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "gemm_tc.cuh"
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
constexpr SplitCost kSplit64 = {0, 0.525, 0.525, 2.6, 0.008};   // 64-row tile pairs, 16 KB stages
constexpr SplitCost kSplit128 = {0, 0.375, 0.375, 2.9, 0.006};  // 128-row tile pairs, 8 KB stages
constexpr SplitCost kSplit256 = {0, 0.59, 0.59, 0.0, 0.059};    // 256-row tile pairs, 8 KB stages (prefill)

struct DeviceState {
    bool ready = false;
    int sms = 0;
    int max_clusters[3] = {0, 0, 0};     // co-resident 2-CTA clusters for tile heights 64, 128, 256 (4-bit)
    int max_clusters_w8[3] = {0, 0, 0};  // the same for the 8-bit kernels
    int max_clusters_sp[2] = {0, 0};     // and for the 2:4 sparse kernels (tile heights 64, 128)
    void* ws = nullptr;
    size_t ws_bytes = 0;
};

constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
long long g_wait_limit_ns = 1000000000LL;

int ceil_div(int a, int b) { return (a + b - 1) / b; }

int norm_group(int K, int G) { return G == -1 ? K : G; }

bool valid_sizes(int K, int N, int G)
{
    if (K <= 0 || N <= 0 || (K % 8) != 0 || (N % 8) != 0) return false;
    return G == 32 || G == 64 || G == 128 || G == K;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

struct Plan {
    int path;     // 2 = per-weight scaling tcgen05 kernel
    int tm;       // rows of X per tile (MMA N)
    int ksub;     // sub-chunks per pipeline stage (64 values of k; 128 for 2:4 sparse codes)
    int xblocks;  // 64-wide blocks of X per stage (the X tensor map's box depth)
    int cluster;  // CTAs per cluster; 2 share each X tile by TMA multicast
    int m_tiles, n_tiles, n_blocks, KC, ng, iters;
    long long total;
    int units;    // work units (clusters)
    int grid;     // CTAs
    size_t ws_bytes;
};

size_t ws_bytes_for(int grid, int tm) { return kPartialsOff + (size_t)2 * grid * tm * kTileN * sizeof(float); }

// max_clusters: how many 2-CTA clusters of this tile height the device holds at
// once (0 = unknown). fmt: the weight format (kFmt*); 8-bit codes run 128-value
// stages at every tile height (16 KB of codes a stage, as 256 values of 4-bit codes).
Plan make_plan(int M, int N, int K, int G, int sms, int max_clusters = 0, int fmt = kFmtW4)
{
    Plan P;
    P.path = 2;
    P.tm = M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
    if (fmt == kFmtW4Sp && P.tm > 128) P.tm = 128;   // sparse stages leave no room for 256-row X tiles
    P.m_tiles = ceil_div(M, P.tm);
    P.n_tiles = ceil_div(N, kTileN);
    P.ksub = (fmt == kFmtW8 || fmt == kFmtW4Sp) ? 2 : P.tm <= 64 ? 4 : 2;
    P.xblocks = fmt == kFmtW4Sp ? 4 : P.ksub;
    // From 64 rows of X up, X is the larger operand per stage: two CTAs on
    // adjacent weight tiles load it once, by multicast.
    P.cluster = P.tm >= 64 ? 2 : 1;
    P.n_blocks = ceil_div(P.n_tiles, P.cluster);
    P.KC = ceil_div(ceil_div(K, kChunkK), kKPad) * kKPad;
    P.iters = P.KC / P.xblocks;
    P.ng = ceil_div(K, G);
    P.total = (long long)P.n_blocks * P.m_tiles * P.iters;
    long long units = (sms < kMaxGrid ? sms : kMaxGrid) / P.cluster;
    if (P.cluster > 1 && max_clusters > 0 && units > max_clusters) units = max_clusters;
    const long long work_tiles = (long long)P.n_blocks * P.m_tiles;
    if (work_tiles < units) {
        // Fewer tiles (or tile pairs) than work units: every tile is cut into the
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
        units = work_tiles * best_s;
    } else {
        // Stream-K over every SM, but a work unit takes at least kMinItersPerCta
        // stages, and with 32 or more rows of X at least a quarter (32 rows) or a
        // half (64 and up) of a tile's stages: the last contributor of a split
        // tile reads every other contributor's partial, which costs about one
        // round trip per 16 rows.
        int min_iters = P.tm >= 64 ? P.iters / 2 : P.tm == 32 ? P.iters / 4 : 0;
        if (min_iters < kMinItersPerCta) min_iters = kMinItersPerCta;
        const long long by_work = (P.total + min_iters - 1) / min_iters;
        if (units > by_work) units = by_work;
    }
    if (units < 1) units = 1;
    P.units = (int)units;
    P.grid = P.units * P.cluster;
    P.ws_bytes = ws_bytes_for(P.grid, P.tm);
    return P;
}

int max_clusters_for(const DeviceState* st, int tm, int fmt = kFmtW4)
{
    if (fmt == kFmtW4Sp) return tm == 64 ? st->max_clusters_sp[0] : tm == 128 ? st->max_clusters_sp[1] : 0;
    const int* mc = fmt == kFmtW8 ? st->max_clusters_w8 : st->max_clusters;
    return tm == 64 ? mc[0] : tm == 128 ? mc[1] : tm == 256 ? mc[2] : 0;
}

// The plan of a shape on this device, with the cluster count of its kernel.
Plan device_plan(const DeviceState* st, int M, int N, int K, int G, int fmt)
{
    const int mc = max_clusters_for(st, make_plan(M, N, K, G, st->sms, 0, fmt).tm, fmt);
    return make_plan(M, N, K, G, st->sms, mc, fmt);
}

// Shared-memory attributes of every variant of one tile shape (epilogue x weight
// format): *mc4 gets the smallest cluster count over the 4-bit variants, *mc8
// over the 8-bit ones.
template <int TM, int KSUB, int CL>
cudaError_t setup_shape(int* mc4, int* mc8, int* mcsp = nullptr)
{
    int mc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    cudaError_t e;
    if ((e = setup_tc<TM, KSUB, CL, false, kFmtW4>(&mc[0])) != cudaSuccess ||
        (e = setup_tc<TM, KSUB, CL, true, kFmtW4>(&mc[1])) != cudaSuccess ||
        (e = setup_tc<TM, KSUB, CL, false, kFmtW4Zp>(&mc[2])) != cudaSuccess ||
        (e = setup_tc<TM, KSUB, CL, true, kFmtW4Zp>(&mc[3])) != cudaSuccess ||
        (e = setup_tc<TM, KSUB, CL, false, kFmtW4Bf16>(&mc[4])) != cudaSuccess ||
        (e = setup_tc<TM, KSUB, CL, true, kFmtW4Bf16>(&mc[5])) != cudaSuccess ||
        (e = setup_tc<TM, 2, CL, false, kFmtW8>(&mc[6])) != cudaSuccess ||
        (e = setup_tc<TM, 2, CL, true, kFmtW8>(&mc[7])) != cudaSuccess)
        return e;
    int m = mc[0];
    for (int i = 1; i < 6; ++i) m = mc[i] < m ? mc[i] : m;
    *mc4 = m;
    *mc8 = mc[6] < mc[7] ? mc[6] : mc[7];
    if constexpr (TM <= 128) {
        int a = 0, b = 0;
        if ((e = setup_tc<TM, 2, CL, false, kFmtW4Sp>(&a)) != cudaSuccess ||
            (e = setup_tc<TM, 2, CL, true, kFmtW4Sp>(&b)) != cudaSuccess)
            return e;
        if (mcsp) *mcsp = a < b ? a : b;
    }
    return cudaSuccess;
}

template <int TM, int KSUB, int CL>
cudaError_t launch_shape(const CUtensorMap& map, const GemmParams& p, bool epi, int fmt, cudaStream_t stream)
{
    switch (fmt) {
        case kFmtW4Zp:
            return epi ? launch_tc<TM, KSUB, CL, true, kFmtW4Zp>(map, p, stream)
                       : launch_tc<TM, KSUB, CL, false, kFmtW4Zp>(map, p, stream);
        case kFmtW8:
            return epi ? launch_tc<TM, 2, CL, true, kFmtW8>(map, p, stream)
                       : launch_tc<TM, 2, CL, false, kFmtW8>(map, p, stream);
        case kFmtW4Bf16:
            return epi ? launch_tc<TM, KSUB, CL, true, kFmtW4Bf16>(map, p, stream)
                       : launch_tc<TM, KSUB, CL, false, kFmtW4Bf16>(map, p, stream);
        case kFmtW4Sp:
            if constexpr (TM <= 128)
                return epi ? launch_tc<TM, 2, CL, true, kFmtW4Sp>(map, p, stream)
                           : launch_tc<TM, 2, CL, false, kFmtW4Sp>(map, p, stream);
            else
                return cudaErrorInvalidValue;   // the plan never picks 256-row tiles for sparse codes
        default:
            return epi ? launch_tc<TM, KSUB, CL, true, kFmtW4>(map, p, stream)
                       : launch_tc<TM, KSUB, CL, false, kFmtW4>(map, p, stream);
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
        int unused = 0;
        int unused8 = 0;
        if ((e = setup_shape<16, 4, 1>(&unused, &unused8)) != cudaSuccess ||
            (e = setup_shape<32, 4, 1>(&unused, &unused8)) != cudaSuccess ||
            (e = setup_shape<64, 4, 2>(&st.max_clusters[0], &st.max_clusters_w8[0], &st.max_clusters_sp[0])) !=
                cudaSuccess ||
            (e = setup_shape<128, 2, 2>(&st.max_clusters[1], &st.max_clusters_w8[1], &st.max_clusters_sp[1])) !=
                cudaSuccess ||
            (e = setup_shape<256, 2, 2>(&st.max_clusters[2], &st.max_clusters_w8[2])) != cudaSuccess)
            return from_cuda(e);
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess) return from_cuda(e);
            if (q != cudaDriverEntryPointSuccess || !fn) return W4A16_ERR_UNSUPPORTED;
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
            if (const char* s = std::getenv("W4A16_WAIT_LIMIT_NS")) g_wait_limit_ns = std::atoll(s);
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

// X as a 3-D view {64, M, K/64} (strides K*2 and 128 bytes) when K is a multiple of
// 64, so one TMA brings a stage's KSUB blocks of 64 columns; else the plain 2-D
// map {K, M}, one TMA per block, with the ragged K edge zero-filled.
bool encode_x_map(CUtensorMap* map, const void* x, int M, int K, int rows, int ksub, bool allow_3d, int* is_3d,
                  bool bf16 = false)
{
    const CUtensorMapDataType dtype = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint32_t estr[3] = {1, 1, 1};
    if (allow_3d && K % kChunkK == 0) {
        cuuint64_t dims[3] = {(cuuint64_t)kChunkK, (cuuint64_t)M, (cuuint64_t)(K / kChunkK)};
        cuuint64_t strides[2] = {(cuuint64_t)K * 2, (cuuint64_t)kChunkK * 2};
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
    cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    cuuint32_t box[2] = {(cuuint32_t)kChunkK, (cuuint32_t)rows};
    CUresult r = g_encode(map, dtype, 2, const_cast<void*>(x), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    *is_3d = 0;
    return r == CUDA_SUCCESS;
}

w4a16_status gemm_impl(const uint16_t* x, const uint32_t* packed, const uint16_t* scales_packed, uint16_t* y, int M,
                       int N, int K, int G, void* ws, size_t ws_bytes, bool own_ws, cudaStream_t stream,
                       const uint16_t* bias = nullptr, const uint16_t* residual = nullptr, int act = 0,
                       int fmt = kFmtW4, const uint8_t* zeros_packed = nullptr)
{
    if ((fmt == kFmtW4Zp) != (zeros_packed != nullptr)) return W4A16_ERR_INVALID_ARG;
    G = norm_group(K, G);
    if (M < 0 || !valid_sizes(K, N, G)) return W4A16_ERR_INVALID_ARG;
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
    p.g_shift = 30;
    if ((G & (G - 1)) == 0) {
        p.g_shift = 0;
        while ((1 << p.g_shift) < G) ++p.g_shift;
    }
    p.n_tiles = P.n_tiles;
    p.m_tiles = P.m_tiles;
    p.KC = fmt == kFmtW4Sp ? P.KC / 2 : P.KC;   // packed chunks per column (128 values of k when sparse)
    p.iters = P.iters;
    p.total_iters = P.total;
    p.grid = P.grid;
    p.cluster = P.cluster;
    p.units = P.units;
    p.n_blocks = P.n_blocks;
    p.wait_limit_ns = g_wait_limit_ns;
    p.bias = reinterpret_cast<const __half*>(bias);
    p.residual = reinterpret_cast<const __half*>(residual);
    p.act = act;

    CUtensorMap map;
    // With one row tile, a box of M rows rounded up to the 8-row swizzle atom is
    // enough: MMA rows past M feed only output columns that are never stored.
    p.x_rows = P.m_tiles == 1 ? ((M + 7) / 8) * 8 : P.tm;
    // Clusters split a stage's X blocks between their CTAs: one 2-D TMA per block.
    if (!encode_x_map(&map, x, M, K, p.x_rows, P.xblocks, P.cluster == 1, &p.x_3d, fmt == kFmtW4Bf16))
        return W4A16_ERR_INVALID_ARG;
    cudaError_t e;
    const bool epi = bias || residual || act != 0;
    switch (P.tm) {
        case 16: e = launch_shape<16, 4, 1>(map, p, epi, fmt, stream); break;
        case 32: e = launch_shape<32, 4, 1>(map, p, epi, fmt, stream); break;
        case 64: e = launch_shape<64, 4, 2>(map, p, epi, fmt, stream); break;
        case 128: e = launch_shape<128, 2, 2>(map, p, epi, fmt, stream); break;
        default: e = launch_shape<256, 2, 2>(map, p, epi, fmt, stream); break;
    }
    return from_cuda(e);
}

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
        const int mc = st ? max_clusters_for(st, make_plan(M, N, K, G, sms, 0, fmt).tm, fmt) : 0;
        const size_t b = make_plan(M, N, K, G, sms, mc, fmt).ws_bytes;
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

w4a16_status w4a16_check_device_status(void* workspace, w4a16_stream_t stream)
{
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return from_cuda(e);
    if (!workspace) {
        DeviceState* st = nullptr;
        w4a16_status rc = device_state(&st);
        if (rc != W4A16_OK) return rc;
        workspace = st->ws;
        if (!workspace) return W4A16_OK;
    }
    int word = 0;
    if ((e = cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess) return from_cuda(e);
    if (word == 0) return W4A16_OK;
    if ((e = cudaMemset(workspace, 0, kPartialsOff)) != cudaSuccess ||
        (e = cudaDeviceSynchronize()) != cudaSuccess)
        return from_cuda(e);
    return W4A16_ERR_TIMEOUT;
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
    *tile_m = P.tm;
    *grid = P.grid;
    return W4A16_OK;
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

}  // namespace

extern "C" w4a16_status w4a16_gemm_noalloc(const uint16_t* x, const uint32_t* packed,
                                           const uint16_t* scales_packed, uint16_t* y, int M, int N, int K,
                                           int group_size, w4a16_stream_t stream)
{
    const int G = norm_group(K, group_size);
    if (M < 0 || !valid_sizes(K, N, G)) return W4A16_ERR_INVALID_ARG;
    if (M == 0) return W4A16_OK;
    DeviceState* st = nullptr;
    w4a16_status rc = device_state(&st);
    if (rc != W4A16_OK) return rc;
    if (device_plan(st, M, N, K, G, kFmtW4).ws_bytes > kNoAllocBytes) return W4A16_ERR_WORKSPACE;
    void* scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc != W4A16_OK) return rc;
    // The error word and the split-K counters must start at zero; the array keeps
    // whatever the previous call left there.
    cudaError_t e = cudaMemsetAsync(scratch, 0, kPartialsOff, reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return from_cuda(e);
    return gemm_impl(x, packed, scales_packed, y, M, N, K, G, scratch, kNoAllocBytes, false,
                     reinterpret_cast<cudaStream_t>(stream));
}

