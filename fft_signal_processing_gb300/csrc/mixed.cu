// Kernel instantiations of the mixed-radix row transform (mixed.cuh) and its entry point.
#include "mixed.cuh"

namespace gbfft {

cudaError_t run_mixed(int mode, int dir, const void* in, void* out, int64_t nrows, int n,
                      const MixedSched& sch, const float2* tw, const float2* ph, int shift_in,
                      int shift_out, float scale, int mmax, int mmajor, cudaStream_t s,
                      int tn1) {
    if (sch.npass < 1 || sch.npass > kMaxMixedPasses) return cudaErrorInvalidValue;
    switch (mode) {
        case BLU_C2C:
            return dir < 0 ? launch_mixed<BLU_C2C, -1>(in, out, nrows, n, sch, tw, ph, shift_in,
                                                       shift_out, scale, mmax, mmajor, 0, s)
                           : launch_mixed<BLU_C2C, +1>(in, out, nrows, n, sch, tw, ph, shift_in,
                                                       shift_out, scale, mmax, mmajor, 0, s);
        case BLU_R2C:
            return launch_mixed<BLU_R2C, -1>(in, out, nrows, n, sch, tw, ph, 0, 0, 1.f, mmax,
                                             mmajor, 0, s);
        case BLU_C2R:
            return launch_mixed<BLU_C2R, +1>(in, out, nrows, n, sch, tw, ph, 0, 0, 1.f, mmax,
                                             mmajor, 0, s);
        case BLU_R2C2:
            return launch_mixed<BLU_R2C2, -1>(in, out, nrows, n, sch, tw, ph, 0, 0, 1.f, mmax,
                                              mmajor, 0, s);
        case BLU_C2R2:
            return launch_mixed<BLU_C2R2, +1>(in, out, nrows, n, sch, tw, ph, 0, 0, 1.f, mmax,
                                              mmajor, 0, s);
        case kMixedRowsT:
            if (tn1 < 2) return cudaErrorInvalidValue;
            return dir < 0 ? launch_mixed<kMixedRowsT, -1>(in, out, nrows, n, sch, tw, ph, 0,
                                                           shift_out, scale, 0, 0, tn1, s)
                           : launch_mixed<kMixedRowsT, +1>(in, out, nrows, n, sch, tw, ph, 0,
                                                           shift_out, scale, 0, 0, tn1, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t run_mixed_cols(int dir, const float2* in, float2* out, int64_t batch, int n1, int n2,
                           const MixedSched& sch, const float2* tw, const float2* hi,
                           const float2* lo, int lobits, const float2* ph, int shift_in,
                           cudaStream_t s) {
    if (sch.npass < 1 || sch.npass > kMaxMixedPasses) return cudaErrorInvalidValue;
    return dir < 0 ? launch_mixed_cols<BLU_C2C, -1>(in, out, batch, n1, n2, sch, tw, hi, lo,
                                                    lobits, ph, shift_in, 0, 0, 0, s)
                   : launch_mixed_cols<BLU_C2C, +1>(in, out, batch, n1, n2, sch, tw, hi, lo,
                                                    lobits, ph, shift_in, 0, 0, 0, s);
}

cudaError_t run_mixed_cols_real(int mode, const void* in, float2* out, int64_t nrows, int n1,
                                int n2, const MixedSched& sch, const float2* tw,
                                const float2* hi, const float2* lo, int lobits, int mmax,
                                int mmajor, cudaStream_t s) {
    if (sch.npass < 1 || sch.npass > kMaxMixedPasses) return cudaErrorInvalidValue;
    const int64_t ntr = (nrows + 1) / 2;
    if (mode == BLU_R2C2)
        return launch_mixed_cols<BLU_R2C2, -1>(in, out, ntr, n1, n2, sch, tw, hi, lo, lobits,
                                               nullptr, 0, nrows, mmax, mmajor, s);
    if (mode == BLU_C2R2)
        return launch_mixed_cols<BLU_C2R2, +1>(in, out, ntr, n1, n2, sch, tw, hi, lo, lobits,
                                               nullptr, 0, nrows, mmax, mmajor, s);
    return cudaErrorInvalidValue;
}

cudaError_t run_mixed_rows_split(const float2* in, float* out, int64_t nrows, int n1, int n2,
                                 const MixedSched& sch, const float2* tw, cudaStream_t s) {
    if (sch.npass < 1 || sch.npass > kMaxMixedPasses || n1 < 2) return cudaErrorInvalidValue;
    const int64_t ntr = (nrows + 1) / 2;
    return launch_mixed<kMixedRowsT2, +1>(in, out, ntr * n1, n2, sch, tw, nullptr, 0, 0, 1.f, 0,
                                          0, n1, s, nrows);
}

cudaError_t run_mixed_unpack(const float2* Y, float2* F, int64_t nrows, int n, int mmax,
                             int mmajor, cudaStream_t s) {
    const int64_t ntr = (nrows + 1) / 2;
    if (ntr <= 0) return cudaSuccess;
    const int64_t xblocks = ((int64_t)mmax + kMixedThreads) / kMixedThreads;
    const unsigned gy = (unsigned)(ntr < 65535 ? ntr : 65535);
    const unsigned gx = (unsigned)(xblocks < 64 ? xblocks : 64);
    k_mixed_unpack<<<dim3(gx, gy, 1), kMixedThreads, 0, s>>>(Y, F, nrows, n, mmax, mmajor);
    return cudaGetLastError();
}

}  // namespace gbfft
