// Real-row analysis (R2C) and synthesis (C2R) kernels, H = N/2 = 2^1 .. 2^14.
#include "kernels.h"
#include "real_kernel.cuh"

namespace gbfft {

template <int LH>
using RealC = FftCfg<LH, rows_log2e(LH), real_log2w(LH), true>;

cudaError_t run_r2c(int log2h, const float* in, float2* out, int64_t nrows, int mmax,
                    int mmajor, const float2* tw, const float2* twr, cudaStream_t s) {
    switch (log2h) {
#define GBFFT_CASE(L) \
    case L: return launch_r2c<RealC<L>>(in, out, nrows, mmax, mmajor, tw, twr, s);
        GBFFT_CASE(1) GBFFT_CASE(2) GBFFT_CASE(3) GBFFT_CASE(4) GBFFT_CASE(5) GBFFT_CASE(6)
        GBFFT_CASE(7) GBFFT_CASE(8) GBFFT_CASE(9) GBFFT_CASE(10) GBFFT_CASE(11) GBFFT_CASE(12)
        GBFFT_CASE(13) GBFFT_CASE(14)
#undef GBFFT_CASE
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t run_c2r(int log2h, const float2* in, float* out, int64_t nrows, int mmax,
                    int mmajor, const float2* tw, const float2* twr, cudaStream_t s) {
    switch (log2h) {
#define GBFFT_CASE(L) \
    case L: return launch_c2r<RealC<L>>(in, out, nrows, mmax, mmajor, tw, twr, s);
        GBFFT_CASE(1) GBFFT_CASE(2) GBFFT_CASE(3) GBFFT_CASE(4) GBFFT_CASE(5) GBFFT_CASE(6)
        GBFFT_CASE(7) GBFFT_CASE(8) GBFFT_CASE(9) GBFFT_CASE(10) GBFFT_CASE(11) GBFFT_CASE(12)
        GBFFT_CASE(13) GBFFT_CASE(14)
#undef GBFFT_CASE
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gbfft
