// Declarations of the per-size entry functions defined by the inst_*.cu translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gbfft {

#define GBFFT_X_ROWS(L)                                                                    \
    cudaError_t rows_entry_##L(int dir, const float2* in, float2* out, int64_t nrows,       \
                               const float2* tw, int flags, int rp, int* err, uint64_t lim, \
                               cudaStream_t s);
#define GBFFT_X_COLS(L) GBFFT_X_COLS_NAMED(L, cols_entry) GBFFT_X_COLS_NAMED(L, cols_tw_entry)
#define GBFFT_X_COLS_NAMED(L, NAME)                                                        \
    cudaError_t NAME##_##L(int dir, const float2* in, float2* out, int64_t count,           \
                               int log2s, const float2* tw, int flags, int ep,              \
                               const float2* hi, const float2* lo, int lowbits, int* err,   \
                               uint64_t lim, cudaStream_t s, const float2* pre);
#define GBFFT_X_ROWS_T(L)                                                                  \
    cudaError_t rows_t_entry_##L(int dir, const float2* in, float2* out, int64_t count,     \
                                 int log2n1, const float2* tw, int flags, int* err,         \
                                 uint64_t lim, cudaStream_t s);
#define GBFFT_X_REAL(L)                                                                    \
    cudaError_t r2c_entry_##L(const float* in, float2* out, int64_t nrows, int mmax,        \
                              int mmajor, const float2* tw, const float2* twr, int flags,   \
                              int* err, uint64_t lim, cudaStream_t s);                      \
    cudaError_t c2r_entry_##L(const float2* in, float* out, int64_t nrows, int mmax,        \
                              int mmajor, const float2* tw, const float2* twr, int flags,   \
                              int* err, uint64_t lim, cudaStream_t s);

#define GBFFT_X_RPAIR(L)                                                                   \
    cudaError_t rpair_entry_##L(bool analysis, const void* in, void* out, int64_t nrows,    \
                                int mmax, int mmajor, const float2* tw, int flags,          \
                                cudaStream_t s);

#define GBFFT_X_BLUESTEIN(L)                                                               \
    cudaError_t bluestein_entry_##L(int mode, const void* in, void* out, int64_t nrows,      \
                                    int n, int mmax, int mmajor, const float2* chirp,       \
                                    const float2* chirp_out, const float2* bhat,            \
                                    const float2* tw, cudaStream_t s);

#define GBFFT_ROWS_SIZES(X) X(0) X(1) X(2) X(3) X(4) X(5) X(6) X(7) X(8) X(9) X(10) X(11) X(12) X(13) X(14)
#define GBFFT_COLS_SIZES(X) X(1) X(2) X(3) X(4) X(5) X(6) X(7) X(8) X(9) X(10) X(11) X(12)
#define GBFFT_ROWS_T_SIZES(X) X(8) X(9) X(10) X(11) X(12)
#define GBFFT_REAL_SIZES(X) X(1) X(2) X(3) X(4) X(5) X(6) X(7) X(8) X(9) X(10) X(11) X(12) X(13) X(14)
#define GBFFT_RPAIR_SIZES(X) X(2) X(3) X(4) X(5) X(6) X(7) X(8) X(9) X(10) X(11) X(12) X(13) X(14)

#define GBFFT_BLUESTEIN_SIZES(X) X(3) X(4) X(5) X(6) X(7) X(8) X(9) X(10) X(11) X(12) X(13) X(14)

GBFFT_ROWS_SIZES(GBFFT_X_ROWS)
GBFFT_BLUESTEIN_SIZES(GBFFT_X_BLUESTEIN)
GBFFT_COLS_SIZES(GBFFT_X_COLS)
GBFFT_ROWS_T_SIZES(GBFFT_X_ROWS_T)
GBFFT_REAL_SIZES(GBFFT_X_REAL)
GBFFT_RPAIR_SIZES(GBFFT_X_RPAIR)

}  // namespace gbfft
