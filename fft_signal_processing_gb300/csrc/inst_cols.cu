// Strided column kernels (2-D column pass; four-step pass 1 with its inter-pass twiddle).
#include "fft_kernel.cuh"
#include "kernels.h"

namespace gbfft {

template <int L, int DIR, bool TW>
static cudaError_t cols_inst(const float2* in, float2* out, int64_t count, int log2s,
                             const float2* tw, int flags, int ep, const float2* hi,
                             const float2* lo, int lowbits, cudaStream_t s) {
    using C = FftCfg<L, cols_log2e(L), cols_log2w(L, 0), false>;
    MapCols<TW> m{count, log2s, L, ep, hi, lo, lowbits};
    return launch_fft<C, DIR, MapCols<TW>>(in, out, m, tw, flags, s);
}

cudaError_t run_cols(int log2l, int dir, const float2* in, float2* out, int64_t count,
                     int log2s, const float2* tw, int flags, int ep, const float2* hi,
                     const float2* lo, int lowbits, cudaStream_t s) {
    const bool twd = hi != nullptr;
    switch (log2l) {
#define GBFFT_CASE(L)                                                                          \
    case L:                                                                                    \
        if (twd)                                                                               \
            return dir < 0 ? cols_inst<L, -1, true>(in, out, count, log2s, tw, flags, ep, hi, \
                                                    lo, lowbits, s)                            \
                           : cols_inst<L, +1, true>(in, out, count, log2s, tw, flags, ep, hi, \
                                                    lo, lowbits, s);                           \
        return dir < 0 ? cols_inst<L, -1, false>(in, out, count, log2s, tw, flags, ep, hi, lo, \
                                                 lowbits, s)                                   \
                       : cols_inst<L, +1, false>(in, out, count, log2s, tw, flags, ep, hi, lo, \
                                                 lowbits, s);
        GBFFT_CASE(1) GBFFT_CASE(2) GBFFT_CASE(3) GBFFT_CASE(4) GBFFT_CASE(5) GBFFT_CASE(6)
        GBFFT_CASE(7) GBFFT_CASE(8) GBFFT_CASE(9) GBFFT_CASE(10) GBFFT_CASE(11) GBFFT_CASE(12)
#undef GBFFT_CASE
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gbfft
