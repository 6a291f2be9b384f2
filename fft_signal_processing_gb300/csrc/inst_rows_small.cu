// One-pass row kernels, 1 <= N <= 2^9.
#include "fft_kernel.cuh"
#include "kernels.h"

namespace gbfft {

template <int L, int DIR>
static cudaError_t rows_inst(const float2* in, float2* out, int64_t nrows, const float2* tw,
                             int flags, int rp, cudaStream_t s) {
    using C = FftCfg<L, rows_log2e(L), rows_log2w(L), true>;
    MapRows m{nrows, L, rp};
    return launch_fft<C, DIR, MapRows>(in, out, m, tw, flags, s);
}

cudaError_t run_rows_small(int log2n, int dir, const float2* in, float2* out, int64_t nrows,
                           const float2* tw, int flags, int rp, cudaStream_t s) {
    switch (log2n) {
#define GBFFT_CASE(L)                                                                \
    case L:                                                                          \
        return dir < 0 ? rows_inst<L, -1>(in, out, nrows, tw, flags, rp, s)          \
                       : rows_inst<L, +1>(in, out, nrows, tw, flags, rp, s);
        GBFFT_CASE(0) GBFFT_CASE(1) GBFFT_CASE(2) GBFFT_CASE(3) GBFFT_CASE(4) GBFFT_CASE(5)
        GBFFT_CASE(6) GBFFT_CASE(7) GBFFT_CASE(8) GBFFT_CASE(9)
#undef GBFFT_CASE
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gbfft
