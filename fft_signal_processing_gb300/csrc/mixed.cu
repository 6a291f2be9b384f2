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
    return dir < 0 ? launch_mixed_cols<-1>(in, out, batch, n1, n2, sch, tw, hi, lo, lobits, ph,
                                           shift_in, s)
                   : launch_mixed_cols<+1>(in, out, batch, n1, n2, sch, tw, hi, lo, lobits, ph,
                                           shift_in, s);
}

}  // namespace gbfft
