// Host-side dispatch into the kernel instantiations (one switch per kernel family), and the
// compile-time launch geometry of every family.  Each run_* function selects the
// instantiation for a log2 size and a direction and enqueues it on `stream`.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "fft_common.cuh"

namespace gbfft {

// ---- launch geometry ------------------------------------------------------------------------
// Largest radix per pass (log2) of each family: radix 64 for rows of 2^9 points and more (two
// passes up to 4096 points: 64 x 64, one shared-memory exchange), radix 16 elsewhere.
__host__ __device__ constexpr int rows_maxrb(int l) { return l >= 9 ? 6 : 4; }
__host__ __device__ constexpr int cols_maxrb(int) { return 4; }
// The real-row core of 2^11 points (4096-point real rows) takes radix 16: a latency-bound
// workload of few rows, where 512 threads per CTA (4 rows, 3 passes) measured 0.056 ms per
// synthesis + analysis of 2048 rows against 0.0675 ms with radix 64 (128 threads).
__host__ __device__ constexpr int real_maxrb(int lh) { return lh >= 9 && lh != 11 ? 6 : 4; }

__host__ __device__ constexpr int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }
__host__ __device__ constexpr int mini(int a, int b) { return a < b ? a : b; }

// log2 of threads per transform
__host__ __device__ constexpr int rows_log2t(int l) { return l - sched_rbits(l, rows_maxrb(l), 0); }
__host__ __device__ constexpr int cols_log2t(int l) { return l - sched_rbits(l, cols_maxrb(l), 0); }
__host__ __device__ constexpr int real_log2t(int lh) { return lh - sched_rbits(lh, real_maxrb(lh), 0); }

// rows per CTA of the plain one-pass kernel: at least 256 threads per CTA
__host__ __device__ constexpr int rows_log2w(int l) { return clampi(8 - rows_log2t(l), 0, 8); }
// transforms per CTA of the strided families: <= 512 threads, <= 2^14 points per CTA,
// at least 2^log2minw transforms (coalescing width), at most 128
__host__ __device__ constexpr int cols_log2w(int l, int log2minw) {
    return clampi(mini(9 - cols_log2t(l), 14 - l), log2minw, 7);
}
// rows per CTA of the real-row path (H-point core): 128 threads, and 4 rows (32-byte runs of
// the m-major spectrum) while the shared memory stays moderate
__host__ __device__ constexpr int real_log2w(int lh) {
    return clampi(7 - real_log2t(lh), lh >= 13 ? 0 : (lh == 12 ? 1 : 2), 7);
}

// Largest sizes of each family.
constexpr int kMaxLog2OnePass = 14;  // 2^14 points * 8.5 B of padded shared memory per row
constexpr int kMaxLog2Strided = 12;  // columns of 2-D images and the four-step passes
constexpr int kMaxLog2RealH = 14;    // real rows of up to 2^15 points

// ---- dispatch -------------------------------------------------------------------------------
// One-pass rows: nrows contiguous rows of 2^log2n points.  row_parity adds (-1)^row to the
// chessboard (2-D row pass).  Sizes 2^5..2^12 run the persistent bulk-copy kernel, whose
// bounded waits report KERR_WAIT_TIMEOUT into *err after limit_ns nanoseconds.
cudaError_t run_rows(int log2n, int dir, const float2* in, float2* out, int64_t nrows,
                     const float2* tw, int flags, int row_parity, int* err, uint64_t limit_ns,
                     cudaStream_t s);

constexpr int kRowsTmaMinLog2 = 5;
constexpr int kRowsTmaMaxLog2 = 12;
constexpr int kRowsTmaStages = 1;  // one stage per CTA: six CTAs per SM at 2^12

// Strided columns: count columns of matrices [2^log2l][2^log2s] stored back to back.
// elem_parity: 1 for the 2-D chessboard (-1)^(row+col), 0 for the four-step one (-1)^col.
// With hi/lo non-NULL, output k1 of column c is multiplied by w_{L*S}^{c*k1} (four-step).
// Columns of 2^7..2^12 points with at least one full tile per matrix run the persistent
// TMA-staged tile kernel (bounded waits reporting into *err, which may be NULL).
// pre (optional, four-step columns of 2^7..2^10 points, inverse): input element q of each
// transform is multiplied by pre[q] on the load.
cudaError_t run_cols(int log2l, int dir, const float2* in, float2* out, int64_t count,
                     int log2s, const float2* tw, int flags, int elem_parity, const float2* hi,
                     const float2* lo, int lowbits, int* err, uint64_t limit_ns, cudaStream_t s,
                     const float2* pre = nullptr);

// Column tiles of the TMA kernel: W = 4096/L columns up to 512 points (at most 64), 8 columns
// at 1024 points and 4 above.  Wide row runs (32-64 bytes) were measured to matter more than
// CTAs per SM at these lengths.  Radix up to 64.
__host__ __device__ constexpr int tile_log2w(int l) { return l <= 9 ? clampi(12 - l, 3, 6) : (l == 10 ? 3 : 2); }
__host__ __device__ constexpr int cols_tma_log2w(int l) { return tile_log2w(l); }
__host__ __device__ constexpr int cols_tma_maxrb(int l) { return l >= 9 ? 6 : 4; }
constexpr int kColsTmaMinLog2 = 7;
constexpr int kColsTmaMaxLog2 = 12;
// the TMA tile kernel serves a column pass iff its tile fits in one matrix row
__host__ __device__ constexpr bool cols_use_tma(int l, int log2s) {
    return l >= kColsTmaMinLog2 && l <= kColsTmaMaxLog2 && log2s >= cols_tma_log2w(l);
}
// twiddle-table schedule (largest radix) of a column pass
__host__ __device__ constexpr int cols_pass_maxrb(int l, int log2s) {
    return cols_use_tma(l, log2s) ? cols_tma_maxrb(l) : cols_maxrb(l);
}

// From 2^11 points (tiles of 64 and 128 KB) the strided passes run the tile kernels that keep
// the stage apart from a half-length exchange buffer, so that the next tile's copy overlaps the
// transform of the current one (measured faster than sharing one buffer at 2^11 and 2^12).
constexpr int kBigTileMinLog2 = 11;
__host__ __device__ constexpr bool cols_use_big(int l, int log2s) {
    return l >= kBigTileMinLog2 && cols_use_tma(l, log2s);
}
__host__ __device__ constexpr bool rowst_use_big(int l) { return l >= kBigTileMinLog2; }

// Four-step pass 2: count rows of 2^log2n points, row tr = k1 + N1*(tr div N1) written
// transposed into X[k1 + N1*k2] of its 2^(log2n1+log2n)-point transform (persistent kernel,
// bulk copies in, tensor stores out; bounded waits report into *err, which may be NULL).
cudaError_t run_rows_t(int log2n, int dir, const float2* in, float2* out, int64_t count,
                       int log2n1, const float2* tw, int flags, int* err, uint64_t limit_ns,
                       cudaStream_t s);

// blocks of W rows as for the column tiles (W <= N1 always holds for the four-step splits),
// radix up to 64
__host__ __device__ constexpr int rowst_log2w(int l) { return tile_log2w(l); }
__host__ __device__ constexpr int rowst_maxrb(int l) { return l >= 9 ? 6 : 4; }

// Rows of any length n that is not a power of two (chirp-z transform through m = 2^log2m
// points, m >= 2n - 1): chirp[j] = c_j (n entries), bhat = FFT_m(conj c)/m (m entries), tw the
// m-point pass tables; chirp multiplies the loads and chirp_out the stores (they differ when a
// shift is folded in).  mode 0: complex rows; 1: real rows -> spectrum m <= mmax (row-major,
// or m-major if mmajor); 2: spectrum -> real rows.
cudaError_t run_bluestein(int log2m, int mode, const void* in, void* out, int64_t nrows, int n,
                          int mmax, int mmajor, const float2* chirp, const float2* chirp_out,
                          const float2* bhat, const float2* tw, cudaStream_t s);
constexpr int kMaxBluesteinN = 8192;  // 2n - 1 <= 2^14: one pass, the m-point row in one CTA
// Radix and rows per CTA of the one-pass chirp-z kernel's m-point transforms.  The kernel does
// two m-point transforms per row and is bound by latency and issue, not HBM.  Light schedules
// (radix 16: more threads, at most 128 registers, two CTAs per SM) serve m = 2^12 and 2^13
// always, and m = 2^9..2^11 for batches too small to give the radix-64 schedule 8 CTAs per SM
// (measured: m = 2^11 large batches 0.74 vs 0.81 ms with radix 64; 2048 real rows 2x faster
// light; m = 2^12, 2^13 20% and 34% faster light).  At m = 2^14 a row's 1024 radix-16 threads
// would leave 64 registers each, so it keeps radix 32.
// Modes of run_bluestein: complex rows; real rows -> spectrum; spectrum -> real rows; the same
// two with two real rows per transform.  BLU_LIGHT (or'ed in) selects the light schedule.
enum : int { BLU_C2C = 0, BLU_R2C = 1, BLU_C2R = 2, BLU_R2C2 = 3, BLU_C2R2 = 4, BLU_LIGHT = 256 };
__host__ __device__ constexpr int blu_maxrb(int l, bool light) {
    return l >= 9 && l <= 13 && (light || l >= 12) ? 4 : rows_maxrb(l);
}
__host__ __device__ constexpr int blu_log2t(int l, bool light) {
    return l - sched_rbits(l, blu_maxrb(l, light), 0);
}
__host__ __device__ constexpr int blu_log2w(int l, bool light) {
    return clampi(8 - blu_log2t(l, light), 0, 8);
}
// Light schedule for a batch of `transforms` m-point transforms (m = 2^l)?
constexpr int64_t kBluLightCtas = 8 * 152;  // 8 CTAs per SM of a 152-SM GB300
__host__ __device__ constexpr bool blu_light(int l, int64_t transforms) {
    return l >= 12 || (transforms >> blu_log2w(l, false)) < kBluLightCtas;
}
__host__ __device__ constexpr int bluestein_log2m(int64_t n) {
    int l = 0;
    while ((int64_t(1) << l) < 2 * n - 1) ++l;
    return l;
}

// Rows of any length kMaxBluesteinN < n <= kMaxBluesteinMpN (not a power of two): the chirp-z
// transform with four-step m-point FFTs over the workspaces A and B (each ntr * m complex64,
// ntr = nrows for complex rows, (nrows + 1) / 2 for real rows, taken two per transform).
// mode: 0 complex rows; 3 real rows -> spectrum; 4 spectrum -> real rows.
struct ChirpMpTables {
    const float2* chirp;      // c_j (with any fftshift folded in), j < n
    const float2* chirp_out;  // c_k for the store (shift and normalisation folded in), k < n
    const float2* bhat;       // FFT_m(conj c)/m, m entries
    const float2* tw_cols;    // pass tables of the m-point four-step column pass
    const float2* tw_rows;    // pass tables of its row pass
    const float2* hi;         // two-level w_m^q table of the inter-pass twiddle
    const float2* lo;
    int lowbits;
};
cudaError_t run_bluestein_mp(int mode, const void* in, void* out, int64_t nrows, int n,
                             int log2m, int mmax, int mmajor, const ChirpMpTables& t, float2* A,
                             float2* B, int* err, uint64_t lim, cudaStream_t s);
constexpr int64_t kMaxBluesteinMpN = int64_t(1) << 20;  // m = 2^21 at most

// Rows of any length 2 <= n <= kMaxMixedN that factors over {2, 3, 5, 7} (and is not a power of
// two): the mixed-radix Stockham kernel (mixed.cuh).  A plan's schedule: radix[p] in
// {2, 3, 4, 5, 7, 8}, span[p] = radix[0]*...*radix[p-1], off[p] the offset of pass p's twiddle
// table ((cos, sin) of 2*pi*m*r/(span*radix) at m*(radix-1) + r-1) in the plan table.
constexpr int kMaxMixedN = 8192;
constexpr int kMaxMixedPasses = 16;
struct MixedSched {
    int npass;
    int radix[kMaxMixedPasses];
    int span[kMaxMixedPasses];
    int off[kMaxMixedPasses];
    // Division by the pass's butterflies per row n/radix and by its span, and by n: x / d is
    // umulhi(x, magic) with magic = ceil(2^32 / d), exact for x * d < 2^32 (every index here
    // is below 2^14 and every divisor at most 2^13); magic 0 stands for d = 1.
    uint32_t qmagic[kMaxMixedPasses];
    uint32_t smagic[kMaxMixedPasses];
    uint32_t nmagic;
};
__host__ __device__ constexpr uint32_t div_magic(uint32_t d) {
    return d <= 1 ? 0u : (uint32_t)((((uint64_t)1 << 32) + d - 1) / d);
}
constexpr int kMixedThreadsHost = 256;  // threads per CTA of the mixed-radix kernel
// Rows per CTA (about 2048 points a CTA: measured faster than 4096, n = 100 and 1000 0.50
// and 0.55 ms against 0.56 and 0.64 ms per 2^26 points) and the two shared-memory buffers
// they take (the pass twiddles stay in global memory, read through L1: staging them in shared
// memory measured no faster at n = 1000 and slower at n = 3000, 0.79 vs 0.66 ms).
__host__ __device__ constexpr int mixed_rows_per_cta(int n) { return n >= 2048 ? 1 : 2048 / n; }
__host__ __device__ constexpr size_t mixed_smem_bytes(int n) {
    return 2 * (size_t)mixed_rows_per_cta(n) * (size_t)n * 8u;
}
static_assert(mixed_smem_bytes(2047) <= mixed_smem_bytes(kMaxMixedN),
              "the launcher's shared-memory limit covers every length");
// mode: BLU_C2C, BLU_R2C, BLU_C2R, BLU_R2C2, BLU_C2R2 (as run_bluestein), or kMixedRowsT (the
// second pass of the four-step form below: nrows = batch*N1 rows of n = N2 points, row
// b*N1 + k1's output k2 stored at b*N1*N2 + k1 + N1*k2; tn1 = N1); dir the sign of the C2C
// transform (the real modes imply theirs).  ph: (cos, sin)(2*pi*(j*h mod N)/N) over the
// transform length N, the fftshift phase applied on the forward load (shift_in) or,
// conjugated, on the inverse store (shift_out); scale multiplies the C2C output.
constexpr int kMixedRowsT = 5;
cudaError_t run_mixed(int mode, int dir, const void* in, void* out, int64_t nrows, int n,
                      const MixedSched& sch, const float2* tw, const float2* ph, int shift_in,
                      int shift_out, float scale, int mmax, int mmajor, cudaStream_t s,
                      int tn1 = 0);

// Complex rows of length kMaxMixedN < n <= kMaxMixedFourStepN whose prime factors are 2, 3, 5
// and 7, as n = N1*N2 with N1 <= kMaxMixedN1 and N2 <= kMaxMixedN: pass 1 (run_mixed_cols)
// transforms the N2 columns of each [N1][N2] transform into a workspace, times w_n^{n2*k1}
// (two-level table hi/lo of w_n, lobits low bits); pass 2 is run_mixed in mode kMixedRowsT.
constexpr int kMaxMixedN1 = 512;
constexpr int kMixedTwLoBits = 10;  // w_n^q = hi[q >> 10] * lo[q & 1023]
constexpr int64_t kMaxMixedFourStepN = int64_t(1) << 20;
// columns per CTA of pass 1: about 2048 points, at least 8 columns (64-byte row runs)
__host__ __device__ constexpr int mixed_cols_per_cta(int n1) {
    return clampi(2048 / n1, 8, 128);
}
__host__ __device__ constexpr size_t mixed_cols_smem_bytes(int n1) {
    return 2 * (size_t)mixed_cols_per_cta(n1) * (size_t)n1 * 8u;
}
cudaError_t run_mixed_cols(int dir, const float2* in, float2* out, int64_t batch, int n1, int n2,
                           const MixedSched& sch, const float2* tw, const float2* hi,
                           const float2* lo, int lobits, const float2* ph, int shift_in,
                           cudaStream_t s);

// Real rows of 2^log2n points, two per n-point complex transform (rows 2p, 2p+1).
cudaError_t run_real_pair(int log2n, bool analysis, const void* in, void* out, int64_t nrows,
                          int mmax, int mmajor, const float2* tw, int flags, cudaStream_t s);
constexpr int kMaxLog2RealPair = 14;

// Real rows of 2^(log2h+1) points.
// flags: KF_INDEX_ONLY (the diagnostic, real rows of 4096 and 2^15 points) or 0.
cudaError_t run_r2c(int log2h, const float* in, float2* out, int64_t nrows, int mmax,
                    int mmajor, const float2* tw, const float2* twr, int flags, int* err,
                    uint64_t limit_ns, cudaStream_t s);
// Real rows with a core of 2^8..2^11 points and an m-major spectrum (even row count) run
// persistent kernels that overlap each tile's copy with the previous tile's transform.
constexpr bool kRealPersistent = true;
cudaError_t run_c2r(int log2h, const float2* in, float* out, int64_t nrows, int mmax,
                    int mmajor, const float2* tw, const float2* twr, int flags, int* err,
                    uint64_t limit_ns, cudaStream_t s);

}  // namespace gbfft
