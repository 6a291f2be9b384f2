// Rows of any length n (not a power of two, n <= 8192): the chirp-z (Bluestein) transform in
// one kernel, one pass over HBM.
//
// With j*k = (j^2 + k^2 - (k-j)^2)/2 the length-n DFT of sign s is a convolution,
//   X_k = c_k * sum_j (x_j c_j) b_{k-j},   c_j = exp(s*pi*i*j^2/n),   b_d = conj(c_d),
// which m-point FFTs (m a power of two, m >= 2n - 1) evaluate exactly on k < n.  One CTA holds
// W rows; for each row the kernel
//   1. loads x_j * c_j for j < n, zero up to m (in the first radix pass's register order),
//   2. runs the forward m-point Stockham passes (the same register/shared-memory machinery as
//      every power-of-two kernel),
//   3. multiplies by bhat = FFT_m(b)/m (a plan table computed in double precision on the host),
//   4. reorders through shared memory into the first pass's order when the first and last
//      radices differ, and runs the inverse m-point passes,
//   5. stores c_k * conv_k for k < n.
// The fftshift is folded into the chirp tables, for odd n as well: the forward transform reads
// with c_j * exp(+2*pi*i*j*h/n), the inverse stores with c_k * exp(-2*pi*i*k*h/n), h = n/2
// rounded down (for even n these factors are the chessboard (-1)^j).  Rows start at any
// 8-byte boundary, so the loads and stores are plain coalesced per-element accesses rather
// than bulk copies.
//
// The same kernel serves band-limited real rows of any length (the direct-sum 'dft' mode of
// "src/sht/wgsl/fourier.ts", dftAnalysWGSL / dftSynthWGSL, for lengths the power-of-two path
// cannot take): analysis (BLU_R2C) loads the real row as complex points with zero imaginary
// part and stores F_m, m <= mmax, into the row-major or m-major spectrum; synthesis (BLU_C2R)
// assembles the Hermitian spectrum on the load (X_0 = Re F_0, X_m = F_m, X_{n-m} = conj F_m
// for 1 <= m <= mmax, other bins 0) and stores the real part of the inverse transform.
// BLU_R2C2 / BLU_C2R2 take two real rows per transform instead (Mota, "High Performance Fourier
// Transforms on GPUs with GLSL", §2.6 Eq. 17-18): analysis transforms y = x1 + i x2 and unpacks
// X1_k = (Y_k + conj Y_{n-k})/2, X2_k = (Y_k - conj Y_{n-k})/(2i) through shared memory;
// synthesis assembles Y_k = X1_k + i X2_k from both Hermitian spectra and stores Re y and Im y.
// Half the transforms of the one-row modes, for the same outputs.
#pragma once

#include "fft_kernel.cuh"
#include "kernels.h"
#include "launch_cache.cuh"

namespace gbfft {


// Shared-memory slots per transform: the padded exchange, and for the two-row analysis the
// n outputs that the unpack reads.
template <class C, int MODE>
__host__ __device__ constexpr int blu_slots() {
    return MODE == BLU_R2C2 ? (C::SROW > C::N ? C::SROW : C::N) : C::SROW;
}

// CTAs per SM the registers must allow: 512 threads per SM (128 registers a thread) for the
// light radix-16 schedules of m >= 2^9, whose registers hold 16 points; no bound otherwise.
template <class C>
__host__ __device__ constexpr int blu_min_ctas() {
    return C::LOG2N >= 9 && C::E <= 16 && C::THREADS <= 512 ? 512 / C::THREADS : 1;
}

template <class C, int MODE>
__global__ void __launch_bounds__(C::THREADS, blu_min_ctas<C>())
    k_bluestein(const void* in_, void* out_, int64_t nrows, int n, int mmax, int mmajor,
                const float2* __restrict__ chirp, const float2* __restrict__ chirp_out,
                const float2* __restrict__ bhat, const float2* __restrict__ tw) {
    static_assert(C::TFAST, "a row's threads are adjacent lanes (coalesced row accesses)");
    constexpr bool PAIR = MODE == BLU_R2C2 || MODE == BLU_C2R2;
    constexpr int SLOTS = blu_slots<C, MODE>();
    extern __shared__ float2 smem[];
    const int w = (int)threadIdx.x / C::T;
    const int t = (int)threadIdx.x % C::T;
    // one-row modes: transform `row` is row `row`; two-row modes: rows 2*row and 2*row + 1 of
    // the nrows real rows (the second absent when nrows is odd)
    const int64_t row = (int64_t)blockIdx.x * C::W + w;
    const int64_t ntr = PAIR ? (nrows + 1) / 2 : nrows;
    const bool active = row < ntr;
    const bool has2 = PAIR && 2 * row + 1 < nrows;
    float2* sb = smem + w * SLOTS;

    constexpr int R0 = C::radix(0);
    constexpr int B0 = C::E / R0;
    constexpr int S0 = C::N / R0;
    constexpr int RL = C::radix(C::NPASS - 1);
    constexpr int BL = C::E / RL;
    constexpr int SL = C::N / RL;

    // element e of the length-n input: a complex row, a real row, or the Hermitian spectrum
    auto load = [&](int e) -> float2 {
        if constexpr (MODE == BLU_C2C) {
            return ldg_stream(static_cast<const float2*>(in_) + row * n + e);
        } else if constexpr (MODE == BLU_R2C) {
            return make_float2(__ldcs(static_cast<const float*>(in_) + row * n + e), 0.f);
        } else if constexpr (MODE == BLU_R2C2) {  // y = x1 + i x2
            const float* x = static_cast<const float*>(in_) + 2 * row * n + e;
            return make_float2(__ldcs(x), has2 ? __ldcs(x + n) : 0.f);
        } else if constexpr (MODE == BLU_C2R2) {  // Y_e = X1_e + i X2_e
            const float2* F = static_cast<const float2*>(in_);
            if (e > mmax && e < n - mmax) return make_float2(0.f, 0.f);
            const int m = e <= mmax ? e : n - e;
            const int64_t r1 = 2 * row;
            float2 f1 = ldg_stream(F + (mmajor ? (int64_t)m * nrows + r1 : r1 * (mmax + 1) + m));
            float2 f2 = make_float2(0.f, 0.f);
            if (has2)
                f2 = ldg_stream(F + (mmajor ? (int64_t)m * nrows + r1 + 1
                                            : (r1 + 1) * (mmax + 1) + m));
            if (e == 0 || 2 * e == n) {  // X_0 and a Nyquist bin: real
                f1.y = 0.f;
                f2.y = 0.f;
            } else if (e > mmax) {  // mirrored bin: conj
                f1.y = -f1.y;
                f2.y = -f2.y;
            }
            return make_float2(f1.x - f2.y, f1.y + f2.x);
        } else {
            const float2* F = static_cast<const float2*>(in_);
            const int m = e <= mmax ? e : n - e;  // bins above n - mmax mirror m = n - e
            if (e > mmax && e < n - mmax) return make_float2(0.f, 0.f);
            const float2 f = ldg_stream(F + (mmajor ? (int64_t)m * nrows + row
                                                    : row * (mmax + 1) + m));
            if (e == 0 || 2 * e == n) return make_float2(f.x, 0.f);  // X_0 and a Nyquist bin: real
            return e <= mmax ? f : make_float2(f.x, -f.y);
        }
    };
    float2 v[C::E];
#pragma unroll
    for (int b = 0; b < B0; ++b) {
        const int j = t + b * C::T;
#pragma unroll
        for (int r = 0; r < R0; ++r) {
            const int e = j + r * S0;
            float2 a = make_float2(0.f, 0.f);
            if (active && e < n) a = cmul(load(e), __ldg(chirp + e));
            v[b * R0 + r] = a;
        }
    }

    run_passes<C, -1, 0>(v, t, sb, tw);  // A = FFT_m(a); element k = j + r*SL in registers

    if constexpr (R0 == RL) {
        // the last pass leaves element j + r*N/R in v[b*R + r]: the first pass's order already
#pragma unroll
        for (int b = 0; b < BL; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < RL; ++r)
                v[b * RL + r] = cmul(v[b * RL + r], __ldg(bhat + j + r * SL));
        }
    } else {
        __syncthreads();  // every thread has read the last exchange
#pragma unroll
        for (int b = 0; b < BL; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < RL; ++r) {
                const int k = j + r * SL;
                sb[spad<C::LP>(k) * C::SS] = cmul(v[b * RL + r], __ldg(bhat + k));
            }
        }
        __syncthreads();
#pragma unroll
        for (int b = 0; b < B0; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < R0; ++r) v[b * R0 + r] = sb[spad<C::LP>(j + r * S0) * C::SS];
        }
    }
    if constexpr (C::NPASS > 1) __syncthreads();  // the buffer becomes the next exchange buffer

    run_passes<C, +1, 0>(v, t, sb, tw);  // conv = IFFT_m(A * bhat)

    if constexpr (MODE == BLU_R2C2) {
        // Y_k = c_k conv_k for k < n into shared memory, then the unpack of both rows
        if constexpr (C::NPASS > 1) __syncthreads();  // the last exchange has been read
#pragma unroll
        for (int b = 0; b < BL; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < RL; ++r) {
                const int k = j + r * SL;
                if (k < n) sb[k] = cmul(v[b * RL + r], __ldg(chirp_out + k));
            }
        }
        __syncthreads();
        if (active) {
            float2* F = static_cast<float2*>(out_);
            const int64_t r1 = 2 * row;
            for (int m = t; m <= mmax; m += C::T) {
                const float2 ym = sb[m], yn = sb[m == 0 ? 0 : n - m];
                float2 f1 = make_float2(0.5f * (ym.x + yn.x), 0.5f * (ym.y - yn.y));
                float2 f2 = make_float2(0.5f * (ym.y + yn.y), 0.5f * (yn.x - ym.x));
                if (m == 0 || 2 * m == n) {  // real bins: drop the rounding residue
                    f1.y = 0.f;
                    f2.y = 0.f;
                }
                stg_stream(F + (mmajor ? (int64_t)m * nrows + r1 : r1 * (mmax + 1) + m), f1);
                if (has2)
                    stg_stream(F + (mmajor ? (int64_t)m * nrows + r1 + 1
                                           : (r1 + 1) * (mmax + 1) + m),
                               f2);
            }
        }
        return;
    }
    const int kend = MODE == BLU_R2C ? mmax + 1 : n;  // outputs kept
    if (active) {
#pragma unroll
        for (int b = 0; b < BL; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < RL; ++r) {
                const int k = j + r * SL;
                if (k < kend) {
                    const float2 y = cmul(v[b * RL + r], __ldg(chirp_out + k));
                    if constexpr (MODE == BLU_C2C) {
                        stg_stream(static_cast<float2*>(out_) + row * n + k, y);
                    } else if constexpr (MODE == BLU_R2C) {
                        // bins 0 and n/2 of a real row are real: drop the rounding residue
                        const float2 f = (k == 0 || 2 * k == n) ? make_float2(y.x, 0.f) : y;
                        stg_stream(static_cast<float2*>(out_) +
                                       (mmajor ? (int64_t)k * nrows + row : row * (mmax + 1) + k),
                                   f);
                    } else if constexpr (MODE == BLU_C2R2) {
                        float* x = static_cast<float*>(out_) + 2 * row * n + k;
                        __stcs(x, y.x);
                        if (has2) __stcs(x + n, y.y);
                    } else {
                        __stcs(static_cast<float*>(out_) + row * n + k, y.x);
                    }
                }
            }
        }
    }
}

template <class C, int MODE>
cudaError_t launch_bluestein(const void* in, void* out, int64_t nrows, int n, int mmax,
                             int mmajor, const float2* chirp, const float2* chirp_out,
                             const float2* bhat, const float2* tw, cudaStream_t stream) {
    auto kern = k_bluestein<C, MODE>;
    constexpr size_t smem = (size_t)blu_slots<C, MODE>() * C::W * sizeof(float2);
    static LaunchCache cache;
    LaunchGeom geo;
    cudaError_t e = cache.get(
        [&](int, LaunchGeom*) {
            return smem > 48 * 1024
                       ? cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              (int)smem)
                       : cudaSuccess;
        },
        &geo);
    if (e != cudaSuccess) return e;
    if (2 * (int64_t)n - 1 > C::N) return cudaErrorInvalidValue;
    const bool pair = MODE == BLU_R2C2 || MODE == BLU_C2R2;
    const int64_t ntr = pair ? (nrows + 1) / 2 : nrows;  // transforms
    const int64_t grid = (ntr + C::W - 1) / C::W;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, C::THREADS, smem, stream>>>(in, out, nrows, n, mmax, mmajor, chirp,
                                                       chirp_out, bhat, tw);
    return cudaGetLastError();
}

}  // namespace gbfft
