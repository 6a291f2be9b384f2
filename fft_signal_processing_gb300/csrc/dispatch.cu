// Run-time dispatch from (family, log2 size) to the per-size entry functions.
#include "inst_entries.h"
#include "cols_tma.cuh"
#include "kernels.h"

namespace gbfft {

// cuTensorMapEncodeTiled, resolved once through the runtime (no link against libcuda).
EncodeTiledFn tensor_map_encoder() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

cudaError_t run_rows(int log2n, int dir, const float2* in, float2* out, int64_t nrows,
                     const float2* tw, int flags, int rp, int* err, uint64_t lim,
                     cudaStream_t s) {
    switch (log2n) {
#define GBFFT_C(L) \
    case L: return rows_entry_##L(dir, in, out, nrows, tw, flags, rp, err, lim, s);
        GBFFT_ROWS_SIZES(GBFFT_C)
#undef GBFFT_C
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t run_cols(int log2l, int dir, const float2* in, float2* out, int64_t count,
                     int log2s, const float2* tw, int flags, int ep, const float2* hi,
                     const float2* lo, int lowbits, int* err, uint64_t lim, cudaStream_t s,
                     const float2* pre) {
    switch (log2l) {
#define GBFFT_C(L)                                                                           \
    case L:                                                                                  \
        return hi ? cols_tw_entry_##L(dir, in, out, count, log2s, tw, flags, ep, hi, lo,     \
                                      lowbits, err, lim, s, pre)                             \
                  : cols_entry_##L(dir, in, out, count, log2s, tw, flags, ep, hi, lo, lowbits, \
                                   err, lim, s, pre);
        GBFFT_COLS_SIZES(GBFFT_C)
#undef GBFFT_C
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t run_rows_t(int log2n, int dir, const float2* in, float2* out, int64_t count,
                       int log2n1, const float2* tw, int flags, int* err, uint64_t lim,
                       cudaStream_t s) {
    switch (log2n) {
#define GBFFT_C(L) \
    case L: return rows_t_entry_##L(dir, in, out, count, log2n1, tw, flags, err, lim, s);
        GBFFT_ROWS_T_SIZES(GBFFT_C)
#undef GBFFT_C
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t run_bluestein(int log2m, int mode, const void* in, void* out, int64_t nrows, int n,
                          int mmax, int mmajor, const float2* chirp, const float2* chirp_out,
                          const float2* bhat, const float2* tw, cudaStream_t s) {
    switch (log2m) {
#define GBFFT_C(L)                                                                          \
    case L:                                                                                 \
        return bluestein_entry_##L(mode, in, out, nrows, n, mmax, mmajor, chirp, chirp_out, \
                                   bhat, tw, s);
        GBFFT_BLUESTEIN_SIZES(GBFFT_C)
#undef GBFFT_C
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t run_real_pair(int log2n, bool analysis, const void* in, void* out, int64_t nrows,
                          int mmax, int mmajor, const float2* tw, int flags, cudaStream_t s) {
    switch (log2n) {
#define GBFFT_C(L) \
    case L: return rpair_entry_##L(analysis, in, out, nrows, mmax, mmajor, tw, flags, s);
        GBFFT_RPAIR_SIZES(GBFFT_C)
#undef GBFFT_C
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t run_r2c(int log2h, const float* in, float2* out, int64_t nrows, int mmax,
                    int mmajor, const float2* tw, const float2* twr, int flags, int* err,
                    uint64_t lim, cudaStream_t s) {
    switch (log2h) {
#define GBFFT_C(L) \
    case L: return r2c_entry_##L(in, out, nrows, mmax, mmajor, tw, twr, flags, err, lim, s);
        GBFFT_REAL_SIZES(GBFFT_C)
#undef GBFFT_C
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t run_c2r(int log2h, const float2* in, float* out, int64_t nrows, int mmax,
                    int mmajor, const float2* tw, const float2* twr, int flags, int* err,
                    uint64_t lim, cudaStream_t s) {
    switch (log2h) {
#define GBFFT_C(L) \
    case L: return c2r_entry_##L(in, out, nrows, mmax, mmajor, tw, twr, flags, err, lim, s);
        GBFFT_REAL_SIZES(GBFFT_C)
#undef GBFFT_C
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gbfft
