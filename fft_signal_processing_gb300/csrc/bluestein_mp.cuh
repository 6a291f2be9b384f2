// Rows of any length 8192 < n <= 2^20 (not a power of two): the chirp-z (Bluestein) transform
// with its two m-point FFTs (m the power of two >= 2n - 1, 2^15 <= m <= 2^21) run by the
// four-step kernels over a workspace, since an m-point row no longer fits one CTA.
//
// With c_j = exp(s*pi*i*j^2/n) and b_d = conj(c_d) the length-n DFT of sign s is
//     X_k = c_k * sum_j (x_j c_j) b_{k-j},
// a cyclic convolution of length m evaluated exactly on k < n (as in bluestein.cuh):
//   1. k_chirp_pre:  A_j = x_j c_j for j < n, 0 for n <= j < m;
//   2. four-step forward FFT_m of A (two passes through a second workspace);
//   3. four-step inverse FFT_m of A * bhat, bhat = FFT_m(b)/m (plan table, double precision
//      on the host), the product taken on the load of its first pass;
//   4. k_chirp_post: X_k = c_k A_k for k < n.
// The fftshift is folded into the chirp tables exactly as in bluestein.cuh.  Band-limited real
// rows take two rows per transform (Mota, "High Performance Fourier Transforms on GPUs with
// GLSL", §2.6 Eq. 17-18): the analysis transforms y = x1 + i x2 and unpacks
// X1_k = (Y_k + conj Y_{n-k})/2, X2_k = (Y_k - conj Y_{n-k})/(2i) in step 4; the synthesis
// assembles Y_k = X1_k + i X2_k from the two Hermitian spectra in step 1 (X_0 = Re F_0,
// X_m = F_m and X_{n-m} = conj F_m for 1 <= m <= mmax, a Nyquist bin real) and stores Re y and
// Im y in step 4.  Steps 1 and 4 are elementwise passes with coalesced accesses along rows.
#pragma once

#include "bluestein.cuh"
#include "fft_common.cuh"
#include "launch_cache.cuh"

namespace gbfft {

constexpr int kChirpThreads = 256;

// Transforms of a batch: one per complex row, one per pair of real rows.
__host__ __device__ inline int64_t chirp_transforms(int mode, int64_t nrows) {
    return mode == BLU_C2C ? nrows : (nrows + 1) / 2;
}

// Step 1.  A = [ntr][m]; e runs over a row's m points.
template <int MODE>
__global__ void __launch_bounds__(kChirpThreads)
    k_chirp_pre(const void* in_, float2* A, int64_t nrows, int n, int m, int mmax, int mmajor,
                const float2* __restrict__ chirp) {
    const int64_t ntr = chirp_transforms(MODE, nrows);
    for (int64_t row = blockIdx.y; row < ntr; row += gridDim.y) {
        const bool has2 = MODE != BLU_C2C && 2 * row + 1 < nrows;
        for (int e = blockIdx.x * kChirpThreads + (int)threadIdx.x; e < m;
             e += gridDim.x * kChirpThreads) {
            float2 a = make_float2(0.f, 0.f);
            if (e < n) {
                if constexpr (MODE == BLU_C2C) {
                    a = ldg_stream(static_cast<const float2*>(in_) + row * n + e);
                } else if constexpr (MODE == BLU_R2C2) {  // y = x1 + i x2
                    const float* x = static_cast<const float*>(in_) + 2 * row * n + e;
                    a = make_float2(__ldcs(x), has2 ? __ldcs(x + n) : 0.f);
                } else {  // BLU_C2R2: Y_e = X1_e + i X2_e
                    if (e <= mmax || e >= n - mmax) {
                        const float2* F = static_cast<const float2*>(in_);
                        const int mm = e <= mmax ? e : n - e;
                        const int64_t r1 = 2 * row;
                        float2 f1 = ldg_stream(F + (mmajor ? (int64_t)mm * nrows + r1
                                                           : r1 * (mmax + 1) + mm));
                        float2 f2 = make_float2(0.f, 0.f);
                        if (has2)
                            f2 = ldg_stream(F + (mmajor ? (int64_t)mm * nrows + r1 + 1
                                                        : (r1 + 1) * (mmax + 1) + mm));
                        if (e == 0 || 2 * e == n) {  // X_0 and a Nyquist bin are real
                            f1.y = 0.f;
                            f2.y = 0.f;
                        } else if (e > mmax) {  // mirrored bin: conj
                            f1.y = -f1.y;
                            f2.y = -f2.y;
                        }
                        a = make_float2(f1.x - f2.y, f1.y + f2.x);
                    }
                }
                a = cmul(a, __ldg(chirp + e));
            }
            stg_stream(A + row * m + e, a);
        }
    }
}

// Step 4.  k runs over the outputs kept: n (complex rows, real synthesis) or mmax + 1 (real
// analysis).
template <int MODE>
__global__ void __launch_bounds__(kChirpThreads)
    k_chirp_post(const float2* A, void* out_, int64_t nrows, int n, int m, int mmax, int mmajor,
                 const float2* __restrict__ chirp_out) {
    const int64_t ntr = chirp_transforms(MODE, nrows);
    const int kend = MODE == BLU_R2C2 ? mmax + 1 : n;
    for (int64_t row = blockIdx.y; row < ntr; row += gridDim.y) {
        const bool has2 = MODE != BLU_C2C && 2 * row + 1 < nrows;
        const float2* a = A + row * m;
        for (int k = blockIdx.x * kChirpThreads + (int)threadIdx.x; k < kend;
             k += gridDim.x * kChirpThreads) {
            const float2 y = cmul(ldg_stream(a + k), __ldg(chirp_out + k));
            if constexpr (MODE == BLU_C2C) {
                stg_stream(static_cast<float2*>(out_) + row * n + k, y);
            } else if constexpr (MODE == BLU_C2R2) {
                float* x = static_cast<float*>(out_) + 2 * row * n + k;
                __stcs(x, y.x);
                if (has2) __stcs(x + n, y.y);
            } else {  // BLU_R2C2: unpack both rows' bin k from Y_k and Y_{n-k}
                const int kn = k == 0 ? 0 : n - k;
                const float2 yn = cmul(ldg_stream(a + kn), __ldg(chirp_out + kn));
                float2 f1 = make_float2(0.5f * (y.x + yn.x), 0.5f * (y.y - yn.y));
                float2 f2 = make_float2(0.5f * (y.y + yn.y), 0.5f * (yn.x - y.x));
                if (k == 0 || 2 * k == n) {  // real bins: drop the rounding residue
                    f1.y = 0.f;
                    f2.y = 0.f;
                }
                float2* F = static_cast<float2*>(out_);
                const int64_t r1 = 2 * row;
                stg_stream(F + (mmajor ? (int64_t)k * nrows + r1 : r1 * (mmax + 1) + k), f1);
                if (has2)
                    stg_stream(F + (mmajor ? (int64_t)k * nrows + r1 + 1 : (r1 + 1) * (mmax + 1) + k),
                               f2);
            }
        }
    }
}

// Grid of an elementwise pass over ntr rows of `len` points: about eight CTAs per SM in all.
inline dim3 chirp_grid(int64_t ntr, int64_t len) {
    static LaunchCache cache;  // the SM count of each device
    LaunchGeom geo;
    if (cache.get([](int dev, LaunchGeom* g) {
            return cudaDeviceGetAttribute(&g->num_sms, cudaDevAttrMultiProcessorCount, dev);
        },
                  &geo) != cudaSuccess)
        geo.num_sms = 1;
    const int64_t target = (int64_t)geo.num_sms * 8;
    const int64_t xblocks = (len + kChirpThreads - 1) / kChirpThreads;
    const int64_t gy = ntr < 65535 ? (ntr < 1 ? 1 : ntr) : 65535;
    int64_t gx = (target + gy - 1) / gy;
    gx = gx < 1 ? 1 : (gx > xblocks ? xblocks : gx);
    return dim3((unsigned)gx, (unsigned)gy, 1u);
}

}  // namespace gbfft
