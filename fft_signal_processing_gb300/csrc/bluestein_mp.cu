// Host sequence of the multi-pass chirp-z transform (bluestein_mp.cuh): chirp premultiply,
// four-step forward FFT, four-step inverse FFT with the filter on its first load, chirp
// postmultiply, all on `s`.
#include "bluestein_mp.cuh"
#include "kernels.h"

namespace gbfft {

cudaError_t run_bluestein_mp(int mode, const void* in, void* out, int64_t nrows, int n,
                             int log2m, int mmax, int mmajor, const ChirpMpTables& t, float2* A,
                             float2* B, int* err, uint64_t lim, cudaStream_t s) {
    const int m = 1 << log2m;
    const int l1 = log2m / 2, l2 = log2m - log2m / 2;  // four-step split of m
    const int64_t ntr = chirp_transforms(mode, nrows);
    const dim3 gm = chirp_grid(ntr, m);
    switch (mode) {
        case BLU_C2C:
            k_chirp_pre<BLU_C2C><<<gm, kChirpThreads, 0, s>>>(in, A, nrows, n, m, mmax, mmajor, t.chirp);
            break;
        case BLU_R2C2:
            k_chirp_pre<BLU_R2C2><<<gm, kChirpThreads, 0, s>>>(in, A, nrows, n, m, mmax, mmajor, t.chirp);
            break;
        case BLU_C2R2:
            k_chirp_pre<BLU_C2R2><<<gm, kChirpThreads, 0, s>>>(in, A, nrows, n, m, mmax, mmajor, t.chirp);
            break;
        default: return cudaErrorInvalidValue;
    }
    cudaError_t e = cudaGetLastError();
    // forward FFT_m: A -> B (columns, times w_m^{n2*k1}) -> A (rows, transposed: natural order)
    if (e == cudaSuccess)
        e = run_cols(l1, -1, A, B, ntr << l2, l2, t.tw_cols, 0, 0, t.hi, t.lo, t.lowbits, err, lim, s);
    if (e == cudaSuccess) e = run_rows_t(l2, -1, B, A, ntr << l1, l1, t.tw_rows, 0, err, lim, s);
    // inverse FFT_m of A * bhat, the filter fused into the first pass's load
    if (e == cudaSuccess)
        e = run_cols(l1, +1, A, B, ntr << l2, l2, t.tw_cols, 0, 0, t.hi, t.lo, t.lowbits, err, lim, s,
                     t.bhat);
    if (e == cudaSuccess) e = run_rows_t(l2, +1, B, A, ntr << l1, l1, t.tw_rows, 0, err, lim, s);
    if (e != cudaSuccess) return e;
    const dim3 go = chirp_grid(ntr, mode == BLU_R2C2 ? mmax + 1 : n);
    switch (mode) {
        case BLU_C2C:
            k_chirp_post<BLU_C2C><<<go, kChirpThreads, 0, s>>>(A, out, nrows, n, m, mmax, mmajor, t.chirp_out);
            break;
        case BLU_R2C2:
            k_chirp_post<BLU_R2C2><<<go, kChirpThreads, 0, s>>>(A, out, nrows, n, m, mmax, mmajor, t.chirp_out);
            break;
        default:
            k_chirp_post<BLU_C2R2><<<go, kChirpThreads, 0, s>>>(A, out, nrows, n, m, mmax, mmajor, t.chirp_out);
            break;
    }
    return cudaGetLastError();
}

}  // namespace gbfft
