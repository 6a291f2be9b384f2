// Four-step pass 2: row transforms with a transposing store.
#include "fft_kernel.cuh"
#include "kernels.h"

namespace gbfft {

template <int L, int DIR>
static cudaError_t rows_t_inst(const float2* in, float2* out, int64_t count, int log2n1,
                               const float2* tw, int flags, cudaStream_t s) {
    using C = FftCfg<L, cols_log2e(L), cols_log2w(L, 2), false>;
    MapRowsT m{count, L, log2n1};
    return launch_fft<C, DIR, MapRowsT>(in, out, m, tw, flags, s);
}

cudaError_t run_rows_t(int log2n, int dir, const float2* in, float2* out, int64_t count,
                       int log2n1, const float2* tw, int flags, cudaStream_t s) {
    switch (log2n) {
#define GBFFT_CASE(L)                                                                \
    case L:                                                                          \
        return dir < 0 ? rows_t_inst<L, -1>(in, out, count, log2n1, tw, flags, s)    \
                       : rows_t_inst<L, +1>(in, out, count, log2n1, tw, flags, s);
        GBFFT_CASE(8) GBFFT_CASE(9) GBFFT_CASE(10) GBFFT_CASE(11) GBFFT_CASE(12)
#undef GBFFT_CASE
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gbfft
