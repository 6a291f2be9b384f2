// Entry points of the mixed-radix four-step transform for band-limited real rows (two rows per
// transform), next to the complex entry points declared in kernels.h, and the launch shape of
// the one-pass kernel.
//
// Rows of up to 2^20 points whose prime factors are 2, 3, 5 and 7 run the mixed-radix passes
// of mixed.cuh as a four-step transform n = N1*N2: k_mixed_cols transforms the columns of each
// [N1][N2] matrix with the twiddle w_n^{n2*k1} on its store, then k_mixed in mode kMixedRowsT
// (or kMixedRowsT2 for the synthesis of real rows) transforms the rows with a transposed store;
// the analysis of real rows ends with k_mixed_unpack.
#pragma once

#include "kernels.h"

namespace gbfft {

constexpr int kMixedRowsT2 = 6;  // run_mixed mode: pass 2 of the real synthesis (mixed.cuh)

// Launch shape of the one-pass kernel: 128 threads and about 1024 points per CTA for rows of
// at most 1024 points in batches of at least 8192 transforms (measured faster there: n = 100
// and 1000 at 0.396 and 0.453 ms against 0.503 and 0.555 ms per 2^26 points with the default
// shape; longer rows and smaller batches measured slower), else 256 threads and about 2048
// points (mixed_rows_per_cta, mixed_smem_bytes).
constexpr int kMixedSmallThreads = 128;
__host__ __device__ constexpr bool mixed_small_cta(int n, int64_t transforms) {
    return n <= 1024 && transforms >= 8192;
}
__host__ __device__ constexpr int mixed_threads_for(bool small) {
    return small ? kMixedSmallThreads : kMixedThreadsHost;
}
__host__ __device__ constexpr int mixed_rows_for(int n, bool small) {
    return small ? (n >= 1024 ? 1 : 1024 / n) : mixed_rows_per_cta(n);
}
__host__ __device__ constexpr size_t mixed_smem_bytes_for(int n, bool small) {
    return 2 * (size_t)mixed_rows_for(n, small) * (size_t)n * 8u;
}
static_assert(mixed_smem_bytes_for(1000, true) <= mixed_smem_bytes_for(1024, true) &&
                  mixed_smem_bytes_for(3, true) <= mixed_smem_bytes_for(1024, true),
              "the small shape's shared-memory limit covers its lengths");

// Pass 1 of the real four-step (mode BLU_R2C2: real rows [nrows][n1*n2] float32 -> workspace;
// BLU_C2R2: spectrum in the plan's layout -> workspace): (nrows + 1) / 2 transforms, the
// column passes and the w_n^{n2*k1} twiddle as run_mixed_cols.
cudaError_t run_mixed_cols_real(int mode, const void* in, float2* out, int64_t nrows, int n1,
                                int n2, const MixedSched& sch, const float2* tw,
                                const float2* hi, const float2* lo, int lobits, int mmax,
                                int mmajor, cudaStream_t s);
// Pass 2 of the real synthesis: the n2-point inverse rows of the workspace, Re and Im of each
// transform's output to its two real rows (out [nrows][n1*n2] float32).
cudaError_t run_mixed_rows_split(const float2* in, float* out, int64_t nrows, int n1, int n2,
                                 const MixedSched& sch, const float2* tw, cudaStream_t s);
// The analysis unpack: Y [(nrows + 1) / 2][n] -> spectrum bins m <= mmax of both rows.
cudaError_t run_mixed_unpack(const float2* Y, float2* F, int64_t nrows, int n, int mmax,
                             int mmajor, cudaStream_t s);

}  // namespace gbfft
