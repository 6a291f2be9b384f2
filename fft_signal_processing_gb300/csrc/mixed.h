// Entry points of the mixed-radix four-step transform for band-limited real rows (two rows per
// transform), next to the complex entry points declared in kernels.h.
#pragma once

#include "kernels.h"

namespace gbfft {

constexpr int kMixedRowsT2 = 6;  // run_mixed mode: pass 2 of the real synthesis (mixed.cuh)

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
