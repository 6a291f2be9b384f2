// Instantiation macros: each kernel family is instantiated per log2 size in a translation unit
// of its own (the radix-64 kernels are large), behind a plain entry function per size that the
// dispatcher (dispatch.cu) selects at run time.
#pragma once

#include "bluestein.cuh"
#include "fft_kernel.cuh"
#include "kernels.h"
#include "real_kernel.cuh"
#include "real_pair.cuh"
#include "cols_tma.cuh"
#include "rows_big.cuh"
#include "rows_tma.cuh"
#include "rowst_tma.cuh"
#include "small_kernel.cuh"
#include "tiles_big.cuh"

namespace gbfft {

// One-pass rows: the small-row kernel up to 2^4, the persistent bulk-copy kernel from 2^5 to
// 2^12, the persistent long-row kernel at 2^13 and 2^14.
template <int L, int DIR>
cudaError_t rows_impl(const float2* in, float2* out, int64_t nrows, const float2* tw, int flags,
                      int rp, int* err, uint64_t lim, cudaStream_t s) {
    if constexpr (L <= 4) {
        (void)tw;
        (void)err;
        (void)lim;
        return launch_small<L, DIR>(in, out, nrows, flags, rp, s);
    } else if constexpr (L >= kRowsTmaMinLog2 && L <= kRowsTmaMaxLog2) {
        return launch_rows_tma<RowsTmaCfg<L, rows_maxrb(L), kRowsTmaStages>, DIR>(
            in, out, nrows, tw, flags, rp, err, lim, s);
    } else {
        // 2^13, 2^14: full-row stage for the next row plus a half-row exchange buffer
        using RC = RowsBigCfg<L, rows_maxrb(L), (L == 13 ? 2 : 1)>;
        return launch_rows_big<RC, DIR>(in, out, nrows, tw, flags, rp, err, lim, s);
    }
}

template <int L, int DIR, bool TW>
cudaError_t cols_impl(const float2* in, float2* out, int64_t count, int log2s, const float2* tw,
                      int flags, int ep, const float2* hi, const float2* lo, int lowbits,
                      int* err, uint64_t lim, cudaStream_t s, const float2* pre) {
    if constexpr (L >= kColsTmaMinLog2 && L <= kColsTmaMaxLog2) {
        if (cols_use_tma(L, log2s)) {  // matrices at least one column tile wide
            if constexpr (L >= kBigTileMinLog2) {
                using RC = ColsBigCfg<L, cols_tma_maxrb(L), cols_tma_log2w(L)>;
                return launch_cols_big<RC, DIR, TW>(in, out, count >> log2s, log2s, tw, flags,
                                                    ep, ColsTwiddle{hi, lo, lowbits}, err, lim,
                                                    s);
            } else {
                using RC = ColsTmaCfg<L, cols_tma_maxrb(L), cols_tma_log2w(L)>;
                return launch_cols_tma<RC, DIR, TW>(in, out, count >> log2s, log2s, tw, flags,
                                                    ep, ColsTwiddle{hi, lo, lowbits, pre}, err,
                                                    lim, s);
            }
        }
    }
    // short columns, and images narrower than a tile: the generic strided kernel
    (void)err;
    (void)lim;
    if (pre) return cudaErrorNotSupported;
    using C = FftCfg<L, cols_maxrb(L), cols_log2w(L, 0), false>;
    MapCols<TW> m{count, log2s, L, ep, hi, lo, lowbits};
    return launch_fft<C, DIR, MapCols<TW>>(in, out, m, tw, flags, s);
}

template <int L, int DIR>
cudaError_t rows_t_impl(const float2* in, float2* out, int64_t count, int log2n1,
                        const float2* tw, int flags, int* err, uint64_t lim, cudaStream_t s) {
    if constexpr (rowst_use_big(L)) {
        using RC = RowsTBigCfg<L, rowst_maxrb(L), rowst_log2w(L)>;
        return launch_rowst_big<RC, DIR>(in, out, count, log2n1, tw, flags, err, lim, s);
    } else {
        using RC = RowsTTmaCfg<L, rowst_maxrb(L), rowst_log2w(L)>;
        return launch_rowst_tma<RC, DIR>(in, out, count, log2n1, tw, flags, err, lim, s);
    }
}

// The chirp-z kernel in each of its modes, for one m-point schedule C.
template <class C>
cudaError_t bluestein_modes(int mode, const void* in, void* out, int64_t nrows, int n, int mmax,
                            int mmajor, const float2* chirp, const float2* chirp_out,
                            const float2* bhat, const float2* tw, cudaStream_t s) {
    switch (mode) {
        case BLU_C2C:
            return launch_bluestein<C, BLU_C2C>(in, out, nrows, n, mmax, mmajor, chirp, chirp_out, bhat, tw, s);
        case BLU_R2C:
            return launch_bluestein<C, BLU_R2C>(in, out, nrows, n, mmax, mmajor, chirp, chirp_out, bhat, tw, s);
        case BLU_C2R:
            return launch_bluestein<C, BLU_C2R>(in, out, nrows, n, mmax, mmajor, chirp, chirp_out, bhat, tw, s);
        case BLU_R2C2:
            return launch_bluestein<C, BLU_R2C2>(in, out, nrows, n, mmax, mmajor, chirp, chirp_out, bhat, tw, s);
        case BLU_C2R2:
            return launch_bluestein<C, BLU_C2R2>(in, out, nrows, n, mmax, mmajor, chirp, chirp_out, bhat, tw, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int LH>
using RealC = FftCfg<LH, real_maxrb(LH), real_log2w(LH), false>;

}  // namespace gbfft

#define GBFFT_DEF_ROWS(L)                                                                      \
    cudaError_t gbfft::rows_entry_##L(int dir, const float2* in, float2* out, int64_t nrows,    \
                                      const float2* tw, int flags, int rp, int* err,            \
                                      uint64_t lim, cudaStream_t s) {                           \
        return dir < 0 ? rows_impl<L, -1>(in, out, nrows, tw, flags, rp, err, lim, s)           \
                       : rows_impl<L, +1>(in, out, nrows, tw, flags, rp, err, lim, s);          \
    }

// Column passes: the four-step variant (with the inter-pass twiddle) and the plain one (2-D)
// are separate entry points so that they can live in separate translation units.
#define GBFFT_DEF_COLS_VARIANT(L, NAME, TWV)                                                   \
    cudaError_t gbfft::NAME##_##L(int dir, const float2* in, float2* out, int64_t count,        \
                                  int log2s, const float2* tw, int flags, int ep,               \
                                  const float2* hi, const float2* lo, int lowbits, int* err,    \
                                  uint64_t lim, cudaStream_t s, const float2* pre) {            \
        return dir < 0 ? cols_impl<L, -1, TWV>(in, out, count, log2s, tw, flags, ep, hi, lo,    \
                                               lowbits, err, lim, s, pre)                       \
                       : cols_impl<L, +1, TWV>(in, out, count, log2s, tw, flags, ep, hi, lo,    \
                                               lowbits, err, lim, s, pre);                      \
    }
#define GBFFT_DEF_COLS_PLAIN(L) GBFFT_DEF_COLS_VARIANT(L, cols_entry, false)
#define GBFFT_DEF_COLS_TW(L) GBFFT_DEF_COLS_VARIANT(L, cols_tw_entry, true)

#define GBFFT_DEF_ROWS_T(L)                                                                    \
    cudaError_t gbfft::rows_t_entry_##L(int dir, const float2* in, float2* out, int64_t count,  \
                                        int log2n1, const float2* tw, int flags, int* err,      \
                                        uint64_t lim, cudaStream_t s) {                         \
        return dir < 0 ? rows_t_impl<L, -1>(in, out, count, log2n1, tw, flags, err, lim, s)     \
                       : rows_t_impl<L, +1>(in, out, count, log2n1, tw, flags, err, lim, s);    \
    }

#define GBFFT_DEF_REAL(L)                                                                      \
    cudaError_t gbfft::r2c_entry_##L(const float* in, float2* out, int64_t nrows, int mmax,     \
                                     int mmajor, const float2* tw, const float2* twr,           \
                                     int flags, int* err, uint64_t lim, cudaStream_t s) {       \
        return launch_r2c<RealC<L>>(in, out, nrows, mmax, mmajor, tw, twr, flags, err, lim, s); \
    }                                                                                           \
    cudaError_t gbfft::c2r_entry_##L(const float2* in, float* out, int64_t nrows, int mmax,     \
                                     int mmajor, const float2* tw, const float2* twr,           \
                                     int flags, int* err, uint64_t lim, cudaStream_t s) {       \
        return launch_c2r<RealC<L>>(in, out, nrows, mmax, mmajor, tw, twr, flags, err, lim,     \
                                    s);                                                         \
    }

// Real rows two per complex transform: the one-pass kernel's geometry for n-point rows.
#define GBFFT_DEF_RPAIR(L)                                                                     \
    cudaError_t gbfft::rpair_entry_##L(bool analysis, const void* in, void* out,                \
                                       int64_t nrows, int mmax, int mmajor, const float2* tw,   \
                                       int flags, cudaStream_t s) {                             \
        using C = FftCfg<L, rows_maxrb(L), rows_log2w(L), true>;                               \
        return launch_real_pair<C>(analysis, in, out, nrows, mmax, mmajor, tw, flags, s);      \
    }

#define GBFFT_DEF_BLUESTEIN(L)                                                                 \
    cudaError_t gbfft::bluestein_entry_##L(int mode, const void* in, void* out, int64_t nrows,  \
                                           int n, int mmax, int mmajor, const float2* chirp,    \
                                           const float2* chirp_out, const float2* bhat,         \
                                           const float2* tw, cudaStream_t s) {                  \
        constexpr bool two = blu_maxrb(L, true) != blu_maxrb(L, false);                          \
        if ((mode & BLU_LIGHT) && two)                                                          \
            return bluestein_modes<FftCfg<L, blu_maxrb(L, true), blu_log2w(L, true), true>>(    \
                mode & ~BLU_LIGHT, in, out, nrows, n, mmax, mmajor, chirp, chirp_out, bhat, tw, s); \
        return bluestein_modes<FftCfg<L, blu_maxrb(L, false), blu_log2w(L, false), true>>(      \
            mode & ~BLU_LIGHT, in, out, nrows, n, mmax, mmajor, chirp, chirp_out, bhat, tw, s);  \
    }
