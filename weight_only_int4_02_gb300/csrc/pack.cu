// Offline repack of INT4 codes, FP16 group scales and (for the asymmetric format)
// 4-bit group zero-points into the tile order the
// tcgen05 kernels stream ("quant_marlin_kernel" (aicassindra.com), "The
// architecture: every piece explained": eight 4-bit values per 32-bit word in a
// permuted order chosen once, offline, so the inner loop needs no shuffles).
//
// Word (((nt*KC + kc)*2 + j)*128 + n_in)*4 + w holds k0 = kc*64 + j*32 + w*8 .. k0+7
// of column n = nt*128 + n_in, with KC = ceil(K/64) rounded up to a multiple of 4
// (a 256-value pipeline stage never runs past the buffer); nibble i holds k0 + 2*(i%4) + i/4, so that the
// magic-number unpack of nibbles (i, i+4) yields the FP16 pair (k, k+1) that
// one 32-bit TMEM column of the MMA's A operand holds. A 64-value chunk of one
// 128-column tile is 4 KB of contiguous words (one bulk copy per pipeline stage);
// within it, the 16 bytes a dequant thread reads for its column are adjacent
// to its neighbours' (conflict-free 128-bit shared loads).
#include <cuda_runtime.h>
#include <stdint.h>

namespace w4a16 {

__global__ void pack_codes_kernel(const uint8_t* __restrict__ codes, uint32_t* __restrict__ packed, int K, int N,
                                  int KC, long long total_words)
{
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total_words;
         idx += (long long)gridDim.x * blockDim.x) {
        const int w = (int)(idx & 3);
        const int n_in = (int)((idx >> 2) & 127);
        const int j = (int)((idx >> 9) & 1);
        const long long rest = idx >> 10;
        const int kc = (int)(rest % KC);
        const int nt = (int)(rest / KC);
        const int n = nt * 128 + n_in;
        const int k0 = kc * 64 + j * 32 + w * 8;
        uint32_t word = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int k = k0 + 2 * (i & 3) + (i >> 2);
            const uint32_t c = (k < K && n < N) ? (uint32_t)(codes[(size_t)k * N + n] & 0xF) : 8u;
            word |= c << (4 * i);
        }
        packed[idx] = word;
    }
}

__global__ void pack_scales_kernel(const uint16_t* __restrict__ scales, uint16_t* __restrict__ out, int N, int ng,
                                   long long total)
{
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int n_in = (int)(idx & 127);
        const long long rest = idx >> 7;
        const int g = (int)(rest % ng);
        const int nt = (int)(rest / ng);
        const int n = nt * 128 + n_in;
        out[idx] = n < N ? scales[(size_t)g * N + n] : (uint16_t)0;
    }
}

// Zero-points: byte (nt*ng + g)*64 + b holds z[g][nt*128 + 2b] (bits 0..3) and
// z[g][nt*128 + 2b + 1] (bits 4..7); columns past N hold 8.
__global__ void pack_zeros_kernel(const uint8_t* __restrict__ zeros, uint8_t* __restrict__ out, int N, int ng,
                                  long long total)
{
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int b = (int)(idx & 63);
        const long long rest = idx >> 6;
        const int g = (int)(rest % ng);
        const int nt = (int)(rest / ng);
        const int n = nt * 128 + 2 * b;
        const uint32_t lo = n < N ? (zeros[(size_t)g * N + n] & 0xFu) : 8u;
        const uint32_t hi = n + 1 < N ? (zeros[(size_t)g * N + n + 1] & 0xFu) : 8u;
        out[idx] = (uint8_t)(lo | (hi << 4));
    }
}

// The GEMM kernels start streaming their packed weights before the kernel ahead
// of them in the stream has finished (programmatic dependent launch; they wait
// for it only before they read X). So the kernel just ahead of a GEMM must not
// write its weights. Each repack therefore ends with this kernel, launched in the
// ordinary way: it starts only once the repack has completed and its writes are
// visible, writes nothing, and is the one a following GEMM may overlap.
__global__ void pack_done_kernel() {}

cudaError_t launch_pack_done(cudaStream_t stream)
{
    pack_done_kernel<<<1, 32, 0, stream>>>();
    return cudaGetLastError();
}

cudaError_t launch_pack_zeros(const uint8_t* zeros, uint8_t* zeros_packed, int N, int n_tiles, int ng, int sms,
                              cudaStream_t stream)
{
    const long long total = (long long)n_tiles * ng * 64;
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    const long long cap = (long long)sms * 16;
    if (blocks > cap) blocks = cap;
    pack_zeros_kernel<<<(unsigned)blocks, threads, 0, stream>>>(zeros, zeros_packed, N, ng, total);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_pack_done(stream);
}

// 8-bit codes (W8A16): byte (((nt*KC + kc)*4 + j4)*128 + n_in)*16 + b holds, for
// word b/4 with k0 = kc*64 + j4*16 + 4*(b/4), the code of k0 + {0, 2, 1, 3}[b%4] in
// column nt*128 + n_in: masking bytes 0 and 2 (1 and 3) of a word gives the FP16
// pair (k, k+1) of one TMEM column; a thread's 16 bytes of a 16-value quarter sit
// next to its neighbours'. Positions outside K x N hold 128 (weight 0).
__global__ void pack_codes_w8_kernel(const uint8_t* __restrict__ codes, uint32_t* __restrict__ packed, int K, int N,
                                     int KC, long long total_words)
{
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total_words;
         idx += (long long)gridDim.x * blockDim.x) {
        const int w = (int)(idx & 3);
        const int n_in = (int)((idx >> 2) & 127);
        const int j4 = (int)((idx >> 9) & 3);
        const long long rest = idx >> 11;
        const int kc = (int)(rest % KC);
        const int nt = (int)(rest / KC);
        const int n = nt * 128 + n_in;
        const int k0 = kc * 64 + j4 * 16 + w * 4;
        uint32_t word = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int k = k0 + ((b & 1) << 1) + (b >> 1);   // bytes 0..3 hold k0 + 0, 2, 1, 3
            const uint32_t c = (k < K && n < N) ? (uint32_t)codes[(size_t)k * N + n] : 128u;
            word |= c << (8 * b);
        }
        packed[idx] = word;
    }
}

// 2:4 sparse 4-bit codes: chunks of 128 k (SC per column), 6144 bytes each at
// (nt*SC + sc)*6144: 4096 bytes of stored codes, word ((b*128 + n_in)*4 + wd)
// holding stored values j0 = b*32 + wd*8 .. +7 of column n_in (nibble i: j0 +
// 2*(i%4) + i/4; stored value j is the code at k = 128*sc + 4*(j/2) + position
// j%2 of its group), then 2048 bytes of position words in tensor-memory lane
// order: word (L*4 + mm), nibble u describes group t = 4*((L%16)/8) + u%4 of the
// MMA's 32 values of k (k = 128*sc + 32*mm + 4t) of column 16*(L/16) + 8*(u/4) +
// L%8, bits 0..1 the first position, bits 2..3 the second. A group stores the
// positions of its codes other than 8, in increasing order, filled up to two with
// the smallest free positions (code 8); a group with more than two codes other
// than 8 keeps its first two and is counted in *violations (if not null).

// Positions (p0 < p1) of group T (k = 4T .. 4T+3) of column n; returns 1 if the
// group holds more than two codes other than 8.
__device__ int sp_group(const uint8_t* __restrict__ codes, int K, int N, int n, int T, int* p0, int* p1)
{
    int pos[2] = {0, 0}, count = 0, taken = 0, violation = 0;
    for (int i = 0; i < 4; ++i) {
        const int k = 4 * T + i;
        if (k < K && n < N && codes[(size_t)k * N + n] != 8) {
            if (count < 2) {
                pos[count++] = i;
                taken |= 1 << i;
            } else {
                violation = 1;
            }
        }
    }
    for (int i = 0; i < 4 && count < 2; ++i)
        if (!(taken & (1 << i))) {
            pos[count++] = i;
            taken |= 1 << i;
        }
    *p0 = min(pos[0], pos[1]);
    *p1 = max(pos[0], pos[1]);
    return violation;
}

__global__ void pack_codes_sp_kernel(const uint8_t* __restrict__ codes, uint8_t* __restrict__ packed, int K, int N,
                                     int SC, long long total, unsigned long long* violations)
{
    for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int L = (int)(idx & 127);
        const long long rest = idx >> 7;
        const int sc = (int)(rest % SC);
        const int nt = (int)(rest / SC);
        uint8_t* chunk = packed + (size_t)rest * 6144;
        uint32_t* cw = reinterpret_cast<uint32_t*>(chunk);
        uint32_t* mw = reinterpret_cast<uint32_t*>(chunk + 4096);
        // stored codes of column L
        const int n = nt * 128 + L;
        uint32_t words[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        unsigned long long bad = 0;
        for (int T = 0; T < 32; ++T) {
            int p0, p1;
            bad += sp_group(codes, K, N, n, sc * 32 + T, &p0, &p1);
            const int pos[2] = {p0, p1};
            for (int sl = 0; sl < 2; ++sl) {
                const int j = 2 * T + sl;
                const int k = 4 * (sc * 32 + T) + pos[sl];
                const uint32_t c = (k < K && n < N) ? (uint32_t)(codes[(size_t)k * N + n] & 0xF) : 8u;
                const int o = j & 7;
                const int nib = (o & 1) * 4 + (o >> 1);   // o = 2*(nib%4) + nib/4
                words[j >> 3] |= c << (4 * nib);
            }
        }
        for (int wi = 0; wi < 8; ++wi) {
            const int b = wi >> 2, wd = wi & 3;
            cw[(b * 128 + L) * 4 + wd] = words[wi];
        }
        if (violations && bad) atomicAdd(violations, bad);
        // position words of lane L
        const int half = (L & 15) >> 3;
        for (int mm = 0; mm < 4; ++mm) {
            uint32_t m = 0;
            for (int u = 0; u < 8; ++u) {
                const int col = nt * 128 + 16 * (L >> 4) + 8 * (u >> 2) + (L & 7);
                const int t = 4 * half + (u & 3);
                int p0, p1;
                sp_group(codes, K, N, col, sc * 32 + mm * 8 + t, &p0, &p1);
                m |= (uint32_t)(p0 | (p1 << 2)) << (4 * u);
            }
            mw[L * 4 + mm] = m;
        }
    }
}

cudaError_t launch_pack_sp(const uint8_t* codes, const uint16_t* scales, uint8_t* packed, uint16_t* scales_packed,
                           int K, int N, int SC, int n_tiles, int ng, int sms, unsigned long long* violations,
                           cudaStream_t stream)
{
    const long long total = (long long)n_tiles * SC * 128;
    const long long selems = (long long)n_tiles * ng * 128;
    const int threads = 128;
    const long long cap = (long long)sms * 32;
    long long blocks = (total + threads - 1) / threads;
    if (blocks > cap) blocks = cap;
    pack_codes_sp_kernel<<<(unsigned)blocks, threads, 0, stream>>>(codes, packed, K, N, SC, total, violations);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    blocks = (selems + 255) / 256;
    if (blocks > cap) blocks = cap;
    pack_scales_kernel<<<(unsigned)blocks, 256, 0, stream>>>(scales, scales_packed, N, ng, selems);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_pack_done(stream);
}

cudaError_t launch_pack_w8(const uint8_t* codes, const uint16_t* scales, uint8_t* packed, uint16_t* scales_packed,
                           int K, int N, int KC, int n_tiles, int ng, int sms, cudaStream_t stream)
{
    const long long words = (long long)n_tiles * KC * 2048;
    const long long selems = (long long)n_tiles * ng * 128;
    const int threads = 256;
    const long long cap = (long long)sms * 16;
    long long blocks = (words + threads - 1) / threads;
    if (blocks > cap) blocks = cap;
    pack_codes_w8_kernel<<<(unsigned)blocks, threads, 0, stream>>>(codes, reinterpret_cast<uint32_t*>(packed), K, N,
                                                                    KC, words);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    blocks = (selems + threads - 1) / threads;
    if (blocks > cap) blocks = cap;
    pack_scales_kernel<<<(unsigned)blocks, threads, 0, stream>>>(scales, scales_packed, N, ng, selems);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_pack_done(stream);
}

cudaError_t launch_pack(const uint8_t* codes, const uint16_t* scales, uint32_t* packed, uint16_t* scales_packed,
                        int K, int N, int KC, int n_tiles, int ng, int sms, cudaStream_t stream)
{
    const long long words = (long long)n_tiles * KC * 1024;
    const long long selems = (long long)n_tiles * ng * 128;
    const int threads = 256;
    long long blocks = (words + threads - 1) / threads;
    const long long cap = (long long)sms * 16;
    if (blocks > cap) blocks = cap;
    pack_codes_kernel<<<(unsigned)blocks, threads, 0, stream>>>(codes, packed, K, N, KC, words);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    blocks = (selems + threads - 1) / threads;
    if (blocks > cap) blocks = cap;
    pack_scales_kernel<<<(unsigned)blocks, threads, 0, stream>>>(scales, scales_packed, N, ng, selems);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_pack_done(stream);
}

}  // namespace w4a16
