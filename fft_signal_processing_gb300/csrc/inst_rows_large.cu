// One-pass row kernels, 2^10 <= N <= 2^14, and the dispatcher of the whole family.
#include "fft_kernel.cuh"
#include "kernels.h"

namespace gbfft {

cudaError_t run_rows_small(int log2n, int dir, const float2* in, float2* out, int64_t nrows,
                           const float2* tw, int flags, int rp, cudaStream_t s);

template <int L, int DIR>
static cudaError_t rows_inst(const float2* in, float2* out, int64_t nrows, const float2* tw,
                             int flags, int rp, cudaStream_t s) {
    using C = FftCfg<L, rows_log2e(L), rows_log2w(L), true>;
    MapRows m{nrows, L, rp};
    return launch_fft<C, DIR, MapRows>(in, out, m, tw, flags, s);
}

cudaError_t run_rows(int log2n, int dir, const float2* in, float2* out, int64_t nrows,
                     const float2* tw, int flags, int rp, cudaStream_t s) {
    switch (log2n) {
#define GBFFT_CASE(L)                                                                \
    case L:                                                                          \
        return dir < 0 ? rows_inst<L, -1>(in, out, nrows, tw, flags, rp, s)          \
                       : rows_inst<L, +1>(in, out, nrows, tw, flags, rp, s);
        GBFFT_CASE(10) GBFFT_CASE(11) GBFFT_CASE(12) GBFFT_CASE(13) GBFFT_CASE(14)
#undef GBFFT_CASE
        default: return run_rows_small(log2n, dir, in, out, nrows, tw, flags, rp, s);
    }
}

}  // namespace gbfft
