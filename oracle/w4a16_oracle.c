/*
 * CPU oracle for the W4A16 weight-only INT4 matmul. TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may load
 * this file's library. Nothing in the CUDA library includes, links or calls it,
 * and it includes nothing from the CUDA library: the two share no code.
 *
 * What it computes (the plain definition, no blocking, no reordering):
 *
 *   w[k][n]   = (q[k][n] - z[k / G][n]) * s[k / G][n]             (dequantisation)
 *   y[m][n]   = sum_{k=0}^{K-1} x[m][k] * w[k][n]   (k ascending, FP64)
 *   abs[m][n] = sum_{k=0}^{K-1} |x[m][k] * w[k][n]|               (tolerance term)
 *
 * Sources: "quant_marlin_kernel" (aicassindra.com), "The architecture: every
 * piece explained": weights are INT4 codes packed eight to a 32-bit word with one
 * FP16 scale per group of weights along the reduction dimension (commonly 128);
 * a thread unpacks the codes to FP16 and multiplies by the group scale; the
 * tensor-core MMA multiplies the dequantised weight tile by the FP16
 * activations. "End-to-end flow": activations (tokens x in-features) times
 * weights (in-features x out-features). The zero-point z is 8 for every group
 * (codes 0..15 map to -8..7) unless a zero-point array is given: the symmetric
 * reading of the pages, which never print a zero-point. The asymmetric form, one
 * integer zero-point 0..15 per (group, column), is the reading of "Low-Precision
 * Quantization Kernels in Production" (llms.blog), section 1, which names AWQ
 * checkpoints (whose 4-bit weights carry a per-group zero-point) among the
 * formats the same kernel family serves.
 *
 * FP16 inputs arrive as IEEE-754 binary16 bit patterns and are decoded by this
 * file's own decoder (sign, 5-bit exponent with bias 15, 10-bit fraction,
 * subnormals). Every product x*(q-z)*s has at most 26 significant bits, so it
 * is exact in FP64; only the k-ascending summation rounds.
 *
 * INT8 codes (the W8A16 format): q in 0..255 with the fixed zero-point 128,
 *   w[k][n] = (q[k][n] - 128) * s[k / G][n]
 * ("Low-Precision Quantization Kernels in Production" (llms.blog), section 1 and
 * its comparison table: the Marlin family serves INT4 and INT8 weights with FP16
 * activations; 128 is the symmetric zero-point of unsigned 8-bit codes, the
 * 8-bit counterpart of the 4-bit format's 8). Products have at most 30
 * significant bits: still exact in FP64.
 *
 * BF16 activations (the *_bf16 entry points): x and s arrive as bfloat16 bit
 * patterns (the upper 16 bits of an IEEE-754 binary32) and are decoded by this
 * file's own bfloat16 decoder; the arithmetic is the same FP64 definition. The
 * pages name BF16 beside FP16 as the 16-bit activation type ("Low-Precision
 * Quantization Kernels in Production" (llms.blog), introduction).
 *
 * The packed-layout functions at the end restate the packed word layout that
 * the library's pack entry point documents (the pages fix only "eight 4-bit
 * values per 32-bit word in a permuted order"; the order itself is free), so
 * that the tests can unpack what the GPU packed and compare it bit for bit.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* IEEE-754 binary16 -> double, from the format's definition. */
double w4o_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);            /* subnormal: 0.f * 2^-14 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25); /* 1.f * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 -> double: sign, 8-bit exponent with bias 127, 7-bit fraction. */
double w4o_bf16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)f, -133);           /* subnormal: 0.f * 2^-126 */
    else if (e == 255)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + f), e - 134); /* 1.f * 2^(e-127) */
    return sign ? -v : v;
}

void w4o_decode_bf16(const uint16_t* h, double* out, size_t count)
{
    for (size_t i = 0; i < count; ++i) out[i] = w4o_bf16_to_double(h[i]);
}

typedef double (*decode_fn)(uint16_t);

void w4o_decode_halves(const uint16_t* h, double* out, size_t count)
{
    for (size_t i = 0; i < count; ++i) out[i] = w4o_half_to_double(h[i]);
}

/* Group index of row k. group_size == K means one group per column. */
static int group_of(int k, int G) { return k / G; }

/* Dequantise column n of the weight matrix into w_col[K]. z is [ceil(K/G)][N]
 * integer zero-points, or NULL for the fixed zero-point zdef (8 for 4-bit codes,
 * 128 for 8-bit codes). */
static void dequant_column(const uint8_t* q, const uint16_t* s, const uint8_t* z, int zdef, decode_fn dec,
                           int K, int N, int G, int n, double* w_col)
{
    for (int k = 0; k < K; ++k) {
        int g = group_of(k, G);
        int code = q[(size_t)k * N + n];
        int zero = z ? z[(size_t)g * N + n] : zdef;
        double scale = dec(s[(size_t)g * N + n]);
        w_col[k] = (double)(code - zero) * scale;
    }
}

/* Full dequantised matrix w[K][N] (FP64), for inspection in tests. */
void w4o_dequant_zp(const uint8_t* q, const uint16_t* s, const uint8_t* z, int K, int N, int G, double* w)
{
    double* col = (double*)malloc(sizeof(double) * (size_t)K);
    for (int n = 0; n < N; ++n) {
        dequant_column(q, s, z, 8, w4o_half_to_double, K, N, G, n, col);
        for (int k = 0; k < K; ++k) w[(size_t)k * N + n] = col[k];
    }
    free(col);
}

void w4o_dequant(const uint8_t* q, const uint16_t* s, int K, int N, int G, double* w)
{
    w4o_dequant_zp(q, s, NULL, K, N, G, w);
}

typedef struct {
    const uint16_t* x; const uint8_t* q; const uint16_t* s; const uint8_t* z; int zdef; decode_fn dec;
    int M, N, K, G;
    const int* rows; int nrows;      /* rows of y to evaluate           */
    const int* cols; int ncols;      /* columns of y to evaluate        */
    double* y; double* absum;        /* [nrows][ncols], may be NULL     */
    int col_begin, col_end;          /* this worker's share of cols     */
    const double* xd;                /* decoded x rows [nrows][K]       */
} job_t;

static void* worker(void* arg)
{
    job_t* j = (job_t*)arg;
    double* w_col = (double*)malloc(sizeof(double) * (size_t)j->K);
    for (int c = j->col_begin; c < j->col_end; ++c) {
        dequant_column(j->q, j->s, j->z, j->zdef, j->dec, j->K, j->N, j->G, j->cols[c], w_col);
        for (int r = 0; r < j->nrows; ++r) {
            const double* xr = j->xd + (size_t)r * j->K;
            double acc = 0.0, acc_abs = 0.0;
            for (int k = 0; k < j->K; ++k) {
                double t = xr[k] * w_col[k];
                acc += t;
                acc_abs += fabs(t);
            }
            j->y[(size_t)r * j->ncols + c] = acc;
            if (j->absum) j->absum[(size_t)r * j->ncols + c] = acc_abs;
        }
    }
    free(w_col);
    return NULL;
}

/*
 * y[r][c] = y_ref[rows[r]][cols[c]] for the listed rows and columns (every
 * element is an independent sum, so a sample of elements is exact for those
 * elements). x is [M][K], q is [K][N] (codes 0..15), s is [ceil(K/G)][N], z is
 * [ceil(K/G)][N] (zero-points 0..15) or NULL for 8.
 * Work is split over `threads` POSIX threads by column; the arithmetic of each
 * element does not depend on the split.
 */
static int gemm_sample_any(const uint16_t* x, const uint8_t* q, const uint16_t* s, const uint8_t* z, int zdef,
                           decode_fn dec, int M, int N, int K, int G,
                           const int* rows, int nrows, const int* cols, int ncols,
                           double* y, double* absum, int threads)
{
    if (M < 0 || N < 0 || K < 0 || G <= 0 || nrows < 0 || ncols < 0) return 1;
    double* xd = (double*)malloc(sizeof(double) * ((size_t)nrows * K + 1));
    for (int r = 0; r < nrows; ++r) {
        if (rows[r] < 0 || rows[r] >= M) { free(xd); return 1; }
        for (int k = 0; k < K; ++k)
            xd[(size_t)r * K + k] = dec(x[(size_t)rows[r] * K + k]);
    }
    for (int c = 0; c < ncols; ++c)
        if (cols[c] < 0 || cols[c] >= N) { free(xd); return 1; }
    if (threads < 1) threads = 1;
    if (threads > ncols) threads = ncols > 0 ? ncols : 1;
    pthread_t* tid = (pthread_t*)malloc(sizeof(pthread_t) * threads);
    job_t* jobs = (job_t*)malloc(sizeof(job_t) * threads);
    for (int t = 0; t < threads; ++t) {
        job_t j = {x, q, s, z, zdef, dec, M, N, K, G, rows, nrows, cols, ncols, y, absum,
                   (int)((long long)ncols * t / threads),
                   (int)((long long)ncols * (t + 1) / threads), xd};
        jobs[t] = j;
    }
    for (int t = 1; t < threads; ++t) pthread_create(&tid[t], NULL, worker, &jobs[t]);
    worker(&jobs[0]);
    for (int t = 1; t < threads; ++t) pthread_join(tid[t], NULL);
    free(jobs); free(tid); free(xd);
    return 0;
}

int w4o_gemm_sample_zp(const uint16_t* x, const uint8_t* q, const uint16_t* s, const uint8_t* z,
                       int M, int N, int K, int G,
                       const int* rows, int nrows, const int* cols, int ncols,
                       double* y, double* absum, int threads)
{
    return gemm_sample_any(x, q, s, z, 8, w4o_half_to_double, M, N, K, G, rows, nrows, cols, ncols, y, absum,
                           threads);
}

/* BF16 activations and scales (bfloat16 bit patterns), 4-bit codes, zero-point 8. */
int w4o_gemm_sample_bf16(const uint16_t* x, const uint8_t* q, const uint16_t* s,
                         int M, int N, int K, int G,
                         const int* rows, int nrows, const int* cols, int ncols,
                         double* y, double* absum, int threads)
{
    return gemm_sample_any(x, q, s, NULL, 8, w4o_bf16_to_double, M, N, K, G, rows, nrows, cols, ncols, y, absum,
                           threads);
}

/* The W8A16 format: q[K][N] are 8-bit codes 0..255, zero-point 128. */
int w4o_gemm_sample_w8(const uint16_t* x, const uint8_t* q, const uint16_t* s,
                       int M, int N, int K, int G,
                       const int* rows, int nrows, const int* cols, int ncols,
                       double* y, double* absum, int threads)
{
    return gemm_sample_any(x, q, s, NULL, 128, w4o_half_to_double, M, N, K, G, rows, nrows, cols, ncols, y, absum,
                           threads);
}

void w4o_dequant_w8(const uint8_t* q, const uint16_t* s, int K, int N, int G, double* w)
{
    double* col = (double*)malloc(sizeof(double) * (size_t)K);
    for (int n = 0; n < N; ++n) {
        dequant_column(q, s, NULL, 128, w4o_half_to_double, K, N, G, n, col);
        for (int k = 0; k < K; ++k) w[(size_t)k * N + n] = col[k];
    }
    free(col);
}

int w4o_gemm_sample(const uint16_t* x, const uint8_t* q, const uint16_t* s,
                    int M, int N, int K, int G,
                    const int* rows, int nrows, const int* cols, int ncols,
                    double* y, double* absum, int threads)
{
    return w4o_gemm_sample_zp(x, q, s, NULL, M, N, K, G, rows, nrows, cols, ncols, y, absum, threads);
}

/* The whole output: y[M][N] and absum[M][N]. */
int w4o_gemm_zp(const uint16_t* x, const uint8_t* q, const uint16_t* s, const uint8_t* z,
                int M, int N, int K, int G, double* y, double* absum, int threads)
{
    int* rows = (int*)malloc(sizeof(int) * (size_t)(M > 0 ? M : 1));
    int* cols = (int*)malloc(sizeof(int) * (size_t)(N > 0 ? N : 1));
    for (int i = 0; i < M; ++i) rows[i] = i;
    for (int i = 0; i < N; ++i) cols[i] = i;
    int rc = w4o_gemm_sample_zp(x, q, s, z, M, N, K, G, rows, M, cols, N, y, absum, threads);
    free(rows); free(cols);
    return rc;
}

int w4o_gemm(const uint16_t* x, const uint8_t* q, const uint16_t* s,
             int M, int N, int K, int G, double* y, double* absum, int threads)
{
    return w4o_gemm_zp(x, q, s, NULL, M, N, K, G, y, absum, threads);
}

/*
 * Packed layout, restated for the round-trip check. Column tiles of 128
 * output features, reduction chunks of 64. For tile nt, chunk kc, half j
 * (32 rows of k), feature n_in within the tile and word w within the half:
 *
 *   word index = (((nt * KC + kc) * 2 + j) * 128 + n_in) * 4 + w,
 *   KC = ceil(K/64) rounded up to a multiple of 4 (K padded to a multiple of 256)
 *   word holds k0 = kc*64 + j*32 + w*8 .. k0+7 of column n = nt*128 + n_in;
 *   nibble i (bits 4i..4i+3) holds k = k0 + 2*(i mod 4) + i/4.
 *
 * Positions with k >= K or n >= N hold code 8 (weight 0).
 * Scales: scales_packed[(nt * ng + g) * 128 + n_in] = s[g][nt*128 + n_in], 0 for n >= N.
 * Zero-points: byte (nt * ng + g) * 64 + b of zeros_packed holds z[g][nt*128 + 2b] in
 * bits 0..3 and z[g][nt*128 + 2b + 1] in bits 4..7; columns n >= N hold 8.
 */
static int ceil_div(int a, int b) { return (a + b - 1) / b; }

static int chunks_per_column(int K) { return ceil_div(ceil_div(K, 64), 4) * 4; }

size_t w4o_packed_words(int K, int N) { return (size_t)ceil_div(N, 128) * chunks_per_column(K) * 1024; }

/* Where (k, n) lives: word index and nibble. */
void w4o_locate(int K, int k, int n, size_t* word, int* nibble)
{
    int KC = chunks_per_column(K);
    int nt = n / 128, n_in = n % 128;
    int kc = k / 64, r = k % 64;
    int j = r / 32, r2 = r % 32;
    int w = r2 / 8, o = r2 % 8;                  /* o = 2*(i mod 4) + i/4 */
    int i = (o % 2) * 4 + o / 2;
    *word = ((((size_t)nt * KC + kc) * 2 + j) * 128 + n_in) * 4 + w;
    *nibble = i;
}

/* Unpack codes[K][N] from packed words; returns the number of padding nibbles != 8. */
long long w4o_unpack(const uint32_t* packed, int K, int N, uint8_t* codes)
{
    int KC = chunks_per_column(K), NT = ceil_div(N, 128);
    long long bad_pad = 0;
    for (int nt = 0; nt < NT; ++nt)
        for (int k = 0; k < KC * 64; ++k)
            for (int n_in = 0; n_in < 128; ++n_in) {
                int n = nt * 128 + n_in;
                size_t word; int nib;
                w4o_locate(K, k, n, &word, &nib);
                int c = (packed[word] >> (4 * nib)) & 0xF;
                if (k < K && n < N) codes[(size_t)k * N + n] = (uint8_t)c;
                else if (c != 8) ++bad_pad;
            }
    return bad_pad;
}

/* The oracle's own pack, used only to check that unpack inverts it. */
void w4o_pack(const uint8_t* codes, int K, int N, uint32_t* packed)
{
    size_t total = w4o_packed_words(K, N);
    for (size_t i = 0; i < total; ++i) packed[i] = 0x88888888u;
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n) {
            size_t word; int nib;
            w4o_locate(K, k, n, &word, &nib);
            packed[word] &= ~(0xFu << (4 * nib));
            packed[word] |= (uint32_t)(codes[(size_t)k * N + n] & 0xF) << (4 * nib);
        }
}

/* Unpack scales[ng][N] from the tile-ordered copy; returns count of nonzero pads. */
long long w4o_unpack_scales(const uint16_t* sp, int ng, int N, uint16_t* s)
{
    int NT = ceil_div(N, 128);
    long long bad_pad = 0;
    for (int nt = 0; nt < NT; ++nt)
        for (int g = 0; g < ng; ++g)
            for (int n_in = 0; n_in < 128; ++n_in) {
                int n = nt * 128 + n_in;
                uint16_t v = sp[((size_t)nt * ng + g) * 128 + n_in];
                if (n < N) s[(size_t)g * N + n] = v;
                else if (v != 0) ++bad_pad;
            }
    return bad_pad;
}

/* Unpack zero-points z[ng][N] from the tile-ordered 4-bit copy; returns the
 * number of padding nibbles that are not 8. */
long long w4o_unpack_zeros(const uint8_t* zp, int ng, int N, uint8_t* z)
{
    int NT = ceil_div(N, 128);
    long long bad_pad = 0;
    for (int nt = 0; nt < NT; ++nt)
        for (int g = 0; g < ng; ++g)
            for (int n_in = 0; n_in < 128; ++n_in) {
                int n = nt * 128 + n_in;
                uint8_t byte = zp[((size_t)nt * ng + g) * 64 + n_in / 2];
                uint8_t v = (uint8_t)((byte >> (4 * (n_in % 2))) & 0xF);
                if (n < N) z[(size_t)g * N + n] = v;
                else if (v != 8) ++bad_pad;
            }
    return bad_pad;
}

/*
 * 8-bit packed layout (W8A16), restated for the round-trip check. Column tiles
 * of 128, reduction chunks of 64 (KC as above), each chunk in four quarters of
 * 16 values. For tile nt, chunk kc, quarter j4, feature n_in and byte b of the
 * column's 16 bytes in that quarter:
 *
 *   byte index = (((nt * KC + kc) * 4 + j4) * 128 + n_in) * 16 + b,
 *   word b/4 holds k0 = kc*64 + j4*16 + 4*(b/4) .. k0+3 of column nt*128 + n_in,
 *   byte b%4 = 0, 1, 2, 3 holds k0 + 0, 2, 1, 3.
 *
 * Positions with k >= K or n >= N hold code 128 (weight 0).
 */
size_t w4o_packed_bytes_w8(int K, int N) { return (size_t)ceil_div(N, 128) * chunks_per_column(K) * 8192; }

size_t w4o_locate_w8(int K, int k, int n)
{
    static const int slot_of_offset[4] = {0, 2, 1, 3};   /* k offset in the word -> byte */
    int KC = chunks_per_column(K);
    int nt = n / 128, n_in = n % 128;
    int kc = k / 64, r = k % 64;
    int j4 = r / 16, r2 = r % 16;
    int b = 4 * (r2 / 4) + slot_of_offset[r2 % 4];
    return ((((size_t)nt * KC + kc) * 4 + j4) * 128 + n_in) * 16 + b;
}

/* Unpack 8-bit codes[K][N]; returns the number of padding bytes that are not 128. */
long long w4o_unpack_w8(const uint8_t* packed, int K, int N, uint8_t* codes)
{
    int KC = chunks_per_column(K), NT = ceil_div(N, 128);
    long long bad_pad = 0;
    for (int nt = 0; nt < NT; ++nt)
        for (int k = 0; k < KC * 64; ++k)
            for (int n_in = 0; n_in < 128; ++n_in) {
                int n = nt * 128 + n_in;
                uint8_t c = packed[w4o_locate_w8(K, k, n)];
                if (k < K && n < N) codes[(size_t)k * N + n] = c;
                else if (c != 128) ++bad_pad;
            }
    return bad_pad;
}

void w4o_pack_w8(const uint8_t* codes, int K, int N, uint8_t* packed)
{
    size_t total = w4o_packed_bytes_w8(K, N);
    memset(packed, 128, total);
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n) packed[w4o_locate_w8(K, k, n)] = codes[(size_t)k * N + n];
}

/*
 * 2:4 sparse 4-bit layout (sparse layout v1), restated for the round-trip check.
 * The weights are the dense 4-bit format whose codes are 2:4 sparse along k: in
 * every aligned group of four k of a column at most two codes differ from 8
 * (weight 0). Only two codes per group are stored, with their 2-bit positions.
 * K is padded to a multiple of 256; chunks of 128 k, SC = Kpad / 128 per column.
 * Chunk (nt, sc) takes 6144 bytes at (nt * SC + sc) * 6144:
 *   codes, 4096 bytes: word ((b * 128 + n_in) * 4 + wd) holds stored values
 *     j0 = b*32 + wd*8 .. j0+7 of column nt*128 + n_in, nibble i holding stored
 *     value j0 + 2*(i mod 4) + i/4;
 *   positions, 2048 bytes after the codes, in the order the sparse tensor-core
 *     MMA reads them from tensor memory (lane L, one 32-bit word per MMA of 32 k):
 *     word (L * 4 + mm), nibble u describes group t = 4*((L mod 16)/8) + u mod 4
 *     (k = sc*128 + mm*32 + 4t .. +3) of column n_in = 16*(L/16) + 8*(u/4) + L mod 8;
 *     bits 0..1 of the nibble hold the position (0..3) of the group's first stored
 *     value, bits 2..3 that of its second, first < second.
 * Stored value j of a chunk is the code at k = sc*128 + 4*(j/2) + (position j%2 of
 * group j/2). A group's stored positions: those of its codes other than 8 in
 * increasing order, filled up to two with the smallest positions not taken (their
 * codes are 8). A group with more than two codes other than 8 (not 2:4) keeps its
 * first two and counts as a violation. Padding (k >= K or n >= N): code 8,
 * positions 0 and 1.
 */
size_t w4o_sp_packed_bytes(int K, int N) { return (size_t)ceil_div(N, 128) * (chunks_per_column(K) / 2) * 6144; }

/* Word (lane) and nibble of the positions of group t (0..7 within an MMA of 32 k)
 * of column n_in (0..127) of a chunk. */
static void sp_position_slot(int n_in, int t, int* lane, int* nibble)
{
    *lane = 16 * (n_in / 16) + 8 * (t / 4) + n_in % 8;
    *nibble = 4 * ((n_in / 8) % 2) + t % 4;
}

/* Stored positions of the group at k = 4T (T-th group) of column n. */
static int group_positions(const uint8_t* codes, int K, int N, int n, int T, int pos[2])
{
    int count = 0, taken[4] = {0, 0, 0, 0};
    int violation = 0;
    for (int i = 0; i < 4; ++i) {
        int k = 4 * T + i;
        if (k < K && n < N && codes[(size_t)k * N + n] != 8) {
            if (count < 2) { pos[count++] = i; taken[i] = 1; }
            else violation = 1;
        }
    }
    for (int i = 0; i < 4 && count < 2; ++i)
        if (!taken[i]) { pos[count++] = i; taken[i] = 1; }
    if (pos[0] > pos[1]) { int t = pos[0]; pos[0] = pos[1]; pos[1] = t; }
    return violation;
}

long long w4o_sp_pack(const uint8_t* codes, int K, int N, uint8_t* packed)
{
    int SC = chunks_per_column(K) / 2, NT = ceil_div(N, 128);
    long long violations = 0;
    memset(packed, 0, w4o_sp_packed_bytes(K, N));
    for (int nt = 0; nt < NT; ++nt)
        for (int sc = 0; sc < SC; ++sc) {
            uint8_t* chunk = packed + ((size_t)nt * SC + sc) * 6144;
            uint32_t* cw = (uint32_t*)chunk;
            uint32_t* mw = (uint32_t*)(chunk + 4096);
            for (int n_in = 0; n_in < 128; ++n_in) {
                int n = nt * 128 + n_in;
                for (int T = 0; T < 32; ++T) {        /* group within the chunk */
                    int pos[2];
                    int Tg = sc * 32 + T;
                    violations += group_positions(codes, K, N, n, Tg, pos);
                    int mm = T / 8, t = T % 8, L, u;
                    sp_position_slot(n_in, t, &L, &u);
                    mw[L * 4 + mm] |= (uint32_t)(pos[0] | (pos[1] << 2)) << (4 * u);
                    for (int s = 0; s < 2; ++s) {
                        int j = 2 * T + s, k = 4 * Tg + pos[s];
                        int c = (k < K && n < N) ? codes[(size_t)k * N + n] : 8;
                        int b = j / 32, wd = (j % 32) / 8, o = j % 8;
                        int nib = (o % 2) * 4 + o / 2;     /* o = 2*(nib mod 4) + nib/4 */
                        cw[(b * 128 + n_in) * 4 + wd] |= (uint32_t)(c & 0xF) << (4 * nib);
                    }
                }
            }
        }
    return violations;
}

/* Dense codes[K][N] (8 where nothing is stored) from the sparse layout; returns the
 * number of malformed groups (positions not increasing) plus padding groups that
 * do not hold code 8 at positions 0 and 1. */
long long w4o_sp_unpack(const uint8_t* packed, int K, int N, uint8_t* codes)
{
    int SC = chunks_per_column(K) / 2, NT = ceil_div(N, 128);
    long long bad = 0;
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n) codes[(size_t)k * N + n] = 8;
    for (int nt = 0; nt < NT; ++nt)
        for (int sc = 0; sc < SC; ++sc) {
            const uint8_t* chunk = packed + ((size_t)nt * SC + sc) * 6144;
            const uint32_t* cw = (const uint32_t*)chunk;
            const uint32_t* mw = (const uint32_t*)(chunk + 4096);
            for (int n_in = 0; n_in < 128; ++n_in) {
                int n = nt * 128 + n_in;
                for (int T = 0; T < 32; ++T) {
                    int mm = T / 8, t = T % 8, L, u;
                    sp_position_slot(n_in, t, &L, &u);
                    uint32_t nib4 = (mw[L * 4 + mm] >> (4 * u)) & 0xF;
                    int pos[2] = {(int)(nib4 & 3), (int)(nib4 >> 2)};
                    int Tg = sc * 32 + T;
                    int pad = (4 * Tg >= K) || n >= N;
                    if (pos[0] >= pos[1]) { ++bad; continue; }
                    for (int s = 0; s < 2; ++s) {
                        int j = 2 * T + s, k = 4 * Tg + pos[s];
                        int b = j / 32, wd = (j % 32) / 8, o = j % 8;
                        int nib = (o % 2) * 4 + o / 2;
                        int c = (cw[(b * 128 + n_in) * 4 + wd] >> (4 * nib)) & 0xF;
                        if (pad) { if (c != 8 || pos[0] != 0 || pos[1] != 1) ++bad; }
                        else codes[(size_t)k * N + n] = (uint8_t)c;
                    }
                }
            }
        }
    return bad;
}
