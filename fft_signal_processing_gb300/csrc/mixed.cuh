// Rows whose length n <= kMaxMixedN factors over {2, 3, 5, 7} (n not a power of two): a
// mixed-radix Stockham transform in one kernel, one pass over HBM, without the chirp-z
// detour (two m-point transforms per row, m >= 2n - 1).
//
// The transform follows the radix-2 Stockham autosort formulation of the WGSL kernels of
// "src/sht/wgsl/fourier.ts" and of the CS598 project page ("Fast Fourier Transform on CPU and
// GPU", the Stockham section), with the radix allowed to change from pass to pass (the
// mixed-radix extension that page and Mota, "High Performance Fourier Transforms on GPUs with
// GLSL", §2.3, name for lengths with other factors).  With n = R_0 R_1 ... R_{P-1} and
// Ns = R_0 ... R_{p-1} the span before pass p (radix R = R_p), every butterfly j < n/R of
// pass p
//   reads      a_r = A[j + r*n/R]                                   (r < R),
//   multiplies a_r by w^r, w = exp(s*2*pi*i*(j mod Ns)/(Ns*R)),
//   transforms y_q = sum_r a_r exp(s*2*pi*i*r*q/R)                   (q < R),
//   writes     B[(j - j mod Ns)*R + j mod Ns + q*Ns] = y_q,
// so that after the last pass B holds X_k in natural order.  A and B are two shared-memory
// buffers of the CTA's W rows; the radix-R butterflies (R in {2, 3, 4, 5, 7, 8}) are
// specialised at compile time and each pass dispatches on its radix.  The pass twiddles come
// from a plan table built in double precision on the host, (cos, sin) of 2*pi*m*r/(Ns*R) for
// m < Ns and 1 <= r < R, the sign applied at use.
//
// Load and store epilogues are those of the one-pass chirp-z kernel (bluestein.cuh): complex
// rows with the fftshift phase exp(+2*pi*i*j*h/n) on the forward load or exp(-2*pi*i*k*h/n) on
// the inverse store (h = n/2 rounded down; the chessboard for even n) and the 1/n of a
// normalised plan on the store; band-limited real rows one per transform (zero imaginary
// part in; Hermitian spectrum X_0 = Re F_0, X_m = F_m, X_{n-m} = conj F_m assembled on the
// load) or two per transform (Mota §2.6 Eq. 17-18: y = x1 + i x2 and the unpack
// X1_k = (Y_k + conj Y_{n-k})/2, X2_k = (Y_k - conj Y_{n-k})/(2i); Y_k = X1_k + i X2_k).
#pragma once

#include "fft_common.cuh"
#include "kernels.h"
#include "launch_cache.cuh"
#include "mixed.h"

namespace gbfft {

constexpr int kMixedThreads = kMixedThreadsHost;

// ---- radix-R DFTs of sign DIR, natural order in and out -------------------------------------
// a * (DIR * i)
template <int DIR>
__device__ __forceinline__ float2 mul_si(float2 a) {
    return DIR < 0 ? make_float2(a.y, -a.x) : make_float2(-a.y, a.x);
}

// cos and sin of 2*pi*q/R for odd R in {3, 5, 7}, 1 <= q <= (R-1)/2 (float roundings of the
// exact values).
template <int R>
__device__ __forceinline__ float odd_cos(int q) {
    if constexpr (R == 3) return -0.5f;
    if constexpr (R == 5) return q == 1 ? 0.30901699437494745f : -0.80901699437494734f;
    if constexpr (R == 7)
        return q == 1 ? 0.62348980185873359f : (q == 2 ? -0.22252093395631434f : -0.90096886790241903f);
    return 0.f;
}
template <int R>
__device__ __forceinline__ float odd_sin(int q) {
    if constexpr (R == 3) return 0.86602540378443865f;
    if constexpr (R == 5) return q == 1 ? 0.95105651629515353f : 0.58778525229247314f;
    if constexpr (R == 7)
        return q == 1 ? 0.78183148246802981f : (q == 2 ? 0.97492791218182361f : 0.43388373911755812f);
    return 0.f;
}

template <int R, int DIR>
__device__ __forceinline__ void dft_small(float2 (&x)[R]) {
    if constexpr (R == 2) {
        const float2 a = x[0], b = x[1];
        x[0] = cadd(a, b);
        x[1] = csub(a, b);
    } else if constexpr (R == 4) {
        const float2 t0 = cadd(x[0], x[2]), t1 = csub(x[0], x[2]);
        const float2 t2 = cadd(x[1], x[3]), t3 = mul_si<DIR>(csub(x[1], x[3]));
        x[0] = cadd(t0, t2);
        x[2] = csub(t0, t2);
        x[1] = cadd(t1, t3);
        x[3] = csub(t1, t3);
    } else if constexpr (R == 8) {
        // two radix-4 DFTs of the even and odd points, then X_k = E_k + w^k O_k,
        // X_{k+4} = E_k - w^k O_k with w = exp(DIR*2*pi*i/8)
        float2 e[4] = {x[0], x[2], x[4], x[6]}, o[4] = {x[1], x[3], x[5], x[7]};
        dft_small<4, DIR>(e);
        dft_small<4, DIR>(o);
        constexpr float h = 0.70710678118654752f;
        const float2 o1 = make_float2(h * (o[1].x - DIR * o[1].y), h * (o[1].y + DIR * o[1].x));
        const float2 o2 = mul_si<DIR>(o[2]);
        const float2 o3 = make_float2(h * (-o[3].x - DIR * o[3].y), h * (-o[3].y + DIR * o[3].x));
        x[0] = cadd(e[0], o[0]);
        x[4] = csub(e[0], o[0]);
        x[1] = cadd(e[1], o1);
        x[5] = csub(e[1], o1);
        x[2] = cadd(e[2], o2);
        x[6] = csub(e[2], o2);
        x[3] = cadd(e[3], o3);
        x[7] = csub(e[3], o3);
    } else {
        // odd R: with a_r = x_r + x_{R-r}, b_r = x_r - x_{R-r} (1 <= r <= (R-1)/2),
        // X_q = x_0 + sum_r a_r cos(2 pi r q/R) + DIR*i sum_r b_r sin(2 pi r q/R), and
        // X_{R-q} the same with the second sum subtracted
        constexpr int H = (R - 1) / 2;
        float2 a[H], b[H];
        float2 s0 = x[0];
#pragma unroll
        for (int r = 1; r <= H; ++r) {
            a[r - 1] = cadd(x[r], x[R - r]);
            b[r - 1] = csub(x[r], x[R - r]);
            s0 = cadd(s0, a[r - 1]);
        }
        float2 y[R];
        y[0] = s0;
#pragma unroll
        for (int q = 1; q <= H; ++q) {
            float2 c = x[0], s = make_float2(0.f, 0.f);
#pragma unroll
            for (int r = 1; r <= H; ++r) {
                int rq = (r * q) % R;  // cos(2 pi rq/R) = cos(2 pi (R-rq)/R), sin changes sign
                const bool neg = rq > H;
                if (neg) rq = R - rq;
                const float cv = odd_cos<R>(rq), sv = neg ? -odd_sin<R>(rq) : odd_sin<R>(rq);
                c = make_float2(fmaf(a[r - 1].x, cv, c.x), fmaf(a[r - 1].y, cv, c.y));
                s = make_float2(fmaf(b[r - 1].x, sv, s.x), fmaf(b[r - 1].y, sv, s.y));
            }
            const float2 is = mul_si<DIR>(s);
            y[q] = cadd(c, is);
            y[R - q] = csub(c, is);
        }
#pragma unroll
        for (int q = 0; q < R; ++q) x[q] = y[q];
    }
}

// x / d for the divisors of a schedule (MixedSched: magic = ceil(2^32/d), 0 for d = 1).
__device__ __forceinline__ int mdiv(int x, uint32_t magic) {
    return magic ? (int)__umulhi((uint32_t)x, magic) : x;
}

// One Stockham pass of radix R over the CTA's W rows (row stride n in both buffers), by a CTA
// of THREADS threads.
template <int R, int DIR, int THREADS>
__device__ __forceinline__ void mixed_pass(const float2* A, float2* B, int n, int W, int Ns,
                                           uint32_t qmagic, uint32_t smagic,
                                           const float2* __restrict__ twp) {
    const int q = n / R;  // butterflies per row
    const int total = W * q;
    for (int idx = (int)threadIdx.x; idx < total; idx += THREADS) {
        const int w = mdiv(idx, qmagic);
        const int j = idx - w * q;
        const float2* a = A + w * n;
        float2* b = B + w * n;
        const int m = j - mdiv(j, smagic) * Ns;
        float2 x[R];
#pragma unroll
        for (int r = 0; r < R; ++r) x[r] = a[j + r * q];
        if (Ns > 1) {
            const float2* t = twp + m * (R - 1);
#pragma unroll
            for (int r = 1; r < R; ++r) x[r] = ctw<DIR>(x[r], __ldg(t + r - 1));
        }
        dft_small<R, DIR>(x);
        const int base = (j - m) * R + m;
#pragma unroll
        for (int r = 0; r < R; ++r) b[base + r * Ns] = x[r];
    }
}

// MODE: BLU_C2C, BLU_R2C, BLU_C2R, BLU_R2C2, BLU_C2R2, or kMixedRowsT: the second pass of the
// mixed-radix four-step transform (rows tr = b*N1 + k1 of n = N2 points; output k2 of the row
// stored at X[b*N1*N2 + k1 + N1*k2], with the inverse fftshift phase of index k1 + N1*k2 and
// the scale; tn1 = N1), or kMixedRowsT2: the same for the synthesis of two real rows per
// transform (Re and Im of X to rows 2b and 2b + 1 of nreal real rows).
// Every pass of the schedule over W rows of n points, A -> B -> A ...; returns the buffer that
// holds the result (every thread's writes visible after the closing barrier).
template <int DIR, int THREADS>
__device__ __forceinline__ float2* mixed_passes(float2* A, float2* B, int n, int W,
                                                const MixedSched& sch,
                                                const float2* __restrict__ tw) {
    for (int p = 0; p < sch.npass; ++p) {
        const float2* twp = tw + sch.off[p];
        const int ns = sch.span[p];
        const uint32_t qm = sch.qmagic[p], sm = sch.smagic[p];
        switch (sch.radix[p]) {
            case 2: mixed_pass<2, DIR, THREADS>(A, B, n, W, ns, qm, sm, twp); break;
            case 3: mixed_pass<3, DIR, THREADS>(A, B, n, W, ns, qm, sm, twp); break;
            case 4: mixed_pass<4, DIR, THREADS>(A, B, n, W, ns, qm, sm, twp); break;
            case 5: mixed_pass<5, DIR, THREADS>(A, B, n, W, ns, qm, sm, twp); break;
            case 7: mixed_pass<7, DIR, THREADS>(A, B, n, W, ns, qm, sm, twp); break;
            default: mixed_pass<8, DIR, THREADS>(A, B, n, W, ns, qm, sm, twp); break;
        }
        __syncthreads();
        float2* t = A;
        A = B;
        B = t;
    }
    return A;
}

template <int MODE, int DIR, int THREADS>
__global__ void __launch_bounds__(THREADS)
    k_mixed(const void* in_, void* out_, int64_t nrows, int n, int W, MixedSched sch,
            const float2* __restrict__ tw, const float2* __restrict__ ph, int shift_in,
            int shift_out, float scale, int mmax, int mmajor, uint32_t wmagic,
            uint32_t kmagic, int tn1, int64_t nreal) {
    constexpr bool PAIR = MODE == BLU_R2C2 || MODE == BLU_C2R2;
    constexpr bool SYN = MODE == BLU_C2R || MODE == BLU_C2R2;
    extern __shared__ float2 smem[];
    float2* A = smem;
    float2* B = smem + W * n;
    const int64_t ntr = PAIR ? (nrows + 1) / 2 : nrows;  // transforms
    const int64_t tr0 = (int64_t)blockIdx.x * W;
    const int tid = (int)threadIdx.x;

    // ---- load: W transforms' inputs into A (w fastest for the m-major spectrum gathers) ----
    const bool wfast_in = SYN && mmajor;
    const uint32_t nm = sch.nmagic;
    // complex rows without a load factor: the CTA's rows are one contiguous run
    constexpr bool CONTIG = MODE == BLU_C2C || MODE == kMixedRowsT || MODE == kMixedRowsT2;
    const bool linear_in = CONTIG && !(MODE == BLU_C2C && shift_in);
    const int cnt = (int)((ntr - tr0 < W ? ntr - tr0 : W) * n);  // points of rows that exist
    if (linear_in) {
        const float2* src = static_cast<const float2*>(in_) + tr0 * n;
#pragma unroll 4
        for (int i = tid; i < W * n; i += THREADS)
            A[i] = i < cnt ? ldg_stream(src + i) : make_float2(0.f, 0.f);
    }
#pragma unroll 4
    for (int idx = linear_in ? W * n : tid; idx < W * n; idx += THREADS) {
        int w, e;
        if (wfast_in) {
            e = mdiv(idx, wmagic);
            w = idx - e * W;
        } else {
            w = mdiv(idx, nm);
            e = idx - w * n;
        }
        const int64_t tr = tr0 + w;
        float2 a = make_float2(0.f, 0.f);
        if (tr < ntr) {
            if constexpr (MODE == kMixedRowsT || MODE == kMixedRowsT2) {
                a = ldg_stream(static_cast<const float2*>(in_) + tr * n + e);
            } else if constexpr (MODE == BLU_C2C) {
                a = ldg_stream(static_cast<const float2*>(in_) + tr * n + e);
                if (shift_in) a = ctw<+1>(a, __ldg(ph + e));
            } else if constexpr (MODE == BLU_R2C) {
                a.x = __ldcs(static_cast<const float*>(in_) + tr * n + e);
            } else if constexpr (MODE == BLU_R2C2) {
                const float* x = static_cast<const float*>(in_) + 2 * tr * n + e;
                a.x = __ldcs(x);
                if (2 * tr + 1 < nrows) a.y = __ldcs(x + n);
            } else if (e <= mmax || e >= n - mmax) {  // Hermitian spectra
                const float2* F = static_cast<const float2*>(in_);
                const int m = e <= mmax ? e : n - e;
                const int64_t r1 = PAIR ? 2 * tr : tr;
                float2 f1 = ldg_stream(F + (mmajor ? (int64_t)m * nrows + r1 : r1 * (mmax + 1) + m));
                float2 f2 = make_float2(0.f, 0.f);
                if (PAIR && r1 + 1 < nrows)
                    f2 = ldg_stream(F + (mmajor ? (int64_t)m * nrows + r1 + 1
                                                : (r1 + 1) * (mmax + 1) + m));
                if (e == 0 || 2 * e == n) {  // X_0 and a Nyquist bin are real
                    f1.y = 0.f;
                    f2.y = 0.f;
                } else if (e > mmax) {  // mirrored bin: conj
                    f1.y = -f1.y;
                    f2.y = -f2.y;
                }
                a = PAIR ? make_float2(f1.x - f2.y, f1.y + f2.x) : f1;
            }
        }
        A[w * n + e] = a;
    }
    __syncthreads();

    A = mixed_passes<DIR, THREADS>(A, B, n, W, sch, tw);

    // ---- store from A ----
    if constexpr (MODE == kMixedRowsT2) {
        // synthesis of two real rows per transform: Re y -> row 2b, Im y -> row 2b + 1 of the
        // nreal rows, at k1 + N1*k2 (tn1 = N1)
        const int64_t nfull = (int64_t)tn1 * n;
        const int64_t b0 = tr0 / tn1;
        const int k10 = (int)(tr0 - b0 * tn1);
#pragma unroll 4
        for (int idx = tid; idx < W * n; idx += THREADS) {
            const int k = mdiv(idx, wmagic), w = idx - k * W;
            const int64_t tr = tr0 + w;
            if (tr >= ntr) continue;
            int k1 = k10 + w;
            int64_t b = b0;
            while (k1 >= tn1) {
                k1 -= tn1;
                ++b;
            }
            const float2 v = A[w * n + k];
            float* xr = static_cast<float*>(out_) + 2 * b * nfull + k1 + (int64_t)tn1 * k;
            __stcs(xr, v.x);
            if (2 * b + 1 < nreal) __stcs(xr + nfull, v.y);
        }
    } else if constexpr (MODE == kMixedRowsT) {
        // consecutive threads take consecutive rows k1 (adjacent outputs) when W > 1
        const int64_t nfull = (int64_t)tn1 * n;
        const int64_t b0 = tr0 / tn1;  // transform and k1 of the CTA's first row
        const int k10 = (int)(tr0 - b0 * tn1);
#pragma unroll 4
        for (int idx = tid; idx < W * n; idx += THREADS) {
            const int k = mdiv(idx, wmagic), w = idx - k * W;
            const int64_t tr = tr0 + w;
            if (tr >= ntr) continue;
            int k1 = k10 + w;
            int64_t b = b0;
            while (k1 >= tn1) {  // rows of the next transform(s)
                k1 -= tn1;
                ++b;
            }
            const int64_t kk = k1 + (int64_t)tn1 * k;  // frequency index within the transform
            float2 y = A[w * n + k];
            if (shift_out) y = ctw<-1>(y, __ldg(ph + kk));
            stg_stream(static_cast<float2*>(out_) + b * nfull + kk,
                       make_float2(y.x * scale, y.y * scale));
        }
    } else if constexpr (MODE == BLU_C2C || MODE == BLU_C2R || MODE == BLU_C2R2) {
        if (MODE == BLU_C2C && !shift_out) {  // one contiguous run, as on the load
            float2* dst = static_cast<float2*>(out_) + tr0 * n;
#pragma unroll 4
            for (int i = tid; i < cnt; i += THREADS) {
                const float2 y = A[i];
                stg_stream(dst + i, make_float2(y.x * scale, y.y * scale));
            }
        }
#pragma unroll 4
        for (int idx = MODE == BLU_C2C && !shift_out ? W * n : tid; idx < W * n; idx += THREADS) {
            const int w = mdiv(idx, nm), k = idx - w * n;
            const int64_t tr = tr0 + w;
            if (tr >= ntr) continue;
            float2 y = A[idx];
            if constexpr (MODE == BLU_C2C) {
                if (shift_out) y = ctw<-1>(y, __ldg(ph + k));
                stg_stream(static_cast<float2*>(out_) + tr * n + k,
                           make_float2(y.x * scale, y.y * scale));
            } else if constexpr (MODE == BLU_C2R) {
                __stcs(static_cast<float*>(out_) + tr * n + k, y.x);
            } else {
                float* x = static_cast<float*>(out_) + 2 * tr * n + k;
                __stcs(x, y.x);
                if (2 * tr + 1 < nrows) __stcs(x + n, y.y);
            }
        }
    } else {  // analysis: bins m <= mmax into the spectrum layout (w fastest when m-major)
        const int nk = mmax + 1;
        float2* F = static_cast<float2*>(out_);
        for (int idx = tid; idx < W * nk; idx += THREADS) {
            const int q = mdiv(idx, mmajor ? wmagic : kmagic);
            const int w = mmajor ? idx - q * W : q;
            const int m = mmajor ? q : idx - q * nk;
            const int64_t tr = tr0 + w;
            if (tr >= ntr) continue;
            const float2 ym = A[w * n + m];
            const int64_t r1 = PAIR ? 2 * tr : tr;
            if constexpr (MODE == BLU_R2C) {
                const float2 f = (m == 0 || 2 * m == n) ? make_float2(ym.x, 0.f) : ym;
                stg_stream(F + (mmajor ? (int64_t)m * nrows + r1 : r1 * nk + m), f);
            } else {
                const float2 yn = A[w * n + (m == 0 ? 0 : n - m)];
                float2 f1 = make_float2(0.5f * (ym.x + yn.x), 0.5f * (ym.y - yn.y));
                float2 f2 = make_float2(0.5f * (ym.y + yn.y), 0.5f * (yn.x - ym.x));
                if (m == 0 || 2 * m == n) {  // real bins: drop the rounding residue
                    f1.y = 0.f;
                    f2.y = 0.f;
                }
                stg_stream(F + (mmajor ? (int64_t)m * nrows + r1 : r1 * nk + m), f1);
                if (r1 + 1 < nrows)
                    stg_stream(F + (mmajor ? (int64_t)m * nrows + r1 + 1 : (r1 + 1) * nk + m), f2);
            }
        }
    }
}

// First pass of the mixed-radix four-step transform of n = N1*N2 points (the four-step split
// the CS598 page names, with both factors over {2, 3, 5, 7}): element n1*N2 + n2 of each
// transform.  CTA (b, t) takes the columns n2 in [t*C, t*C + C) of transform b: it loads the
// [N1][C] tile with coalesced row runs (the forward fftshift phase of index n1*N2 + n2 on the
// load) into C rows of N1 points in shared memory, runs the N1-point passes, and writes output
// (k1, n2) times w_n^{n2*k1} to out[b*n + k1*N2 + n2].  w_n^q = hi[q >> lobits] * lo[q & mask]
// (plan tables, (cos, sin) of the positive angle, the sign applied at use).
// MODE BLU_C2C: complex rows (in: [batch][n] complex64).  Band-limited real rows, two per
// transform b (rows 2b, 2b+1 of nrows): BLU_R2C2 loads y = x1 + i x2 (in: [nrows][n] float32);
// BLU_C2R2 assembles Y_j = X1_j + i X2_j from the two Hermitian spectra (in: the spectrum, in
// the plan's layout; X_0 and a Nyquist bin real, X_{n-m} = conj F_m).
template <int MODE, int DIR>
__global__ void __launch_bounds__(kMixedThreads)
    k_mixed_cols(const void* in_, float2* out, int n1, int n2, int C, uint32_t cmagic,
                 int64_t tiles, MixedSched sch, const float2* __restrict__ tw,
                 const float2* __restrict__ hi, const float2* __restrict__ lo, int lobits,
                 const float2* __restrict__ ph, int shift_in, int64_t nrows, int mmax,
                 int mmajor) {
    extern __shared__ float2 smem[];
    float2* A = smem;
    float2* B = smem + C * n1;
    const int64_t b = blockIdx.x / tiles;
    const int c0 = (int)(blockIdx.x - b * tiles) * C;
    const int64_t n = (int64_t)n1 * n2;
    float2* y = out + b * n;
    const int tid = (int)threadIdx.x;
    const int64_t r1 = 2 * b;  // real modes: the transform's first row
    const bool has2 = r1 + 1 < nrows;
#pragma unroll 4
    for (int idx = tid; idx < C * n1; idx += kMixedThreads) {
        const int r = mdiv(idx, cmagic), c = idx - r * C;
        float2 a = make_float2(0.f, 0.f);
        if (c0 + c < n2) {
            const int64_t j = (int64_t)r * n2 + c0 + c;
            if constexpr (MODE == BLU_C2C) {
                a = ldg_stream(static_cast<const float2*>(in_) + b * n + j);
                if (shift_in) a = ctw<+1>(a, __ldg(ph + j));
            } else if constexpr (MODE == BLU_R2C2) {
                const float* xf = static_cast<const float*>(in_) + r1 * n + j;
                a.x = __ldcs(xf);
                if (has2) a.y = __ldcs(xf + n);
            } else if (j <= mmax || j >= n - mmax) {  // BLU_C2R2
                const float2* F = static_cast<const float2*>(in_);
                const int64_t m = j <= mmax ? j : n - j;
                float2 f1 = ldg_stream(F + (mmajor ? m * nrows + r1 : r1 * (mmax + 1) + m));
                float2 f2 = make_float2(0.f, 0.f);
                if (has2)
                    f2 = ldg_stream(F + (mmajor ? m * nrows + r1 + 1 : (r1 + 1) * (mmax + 1) + m));
                if (j == 0 || 2 * j == n) {  // X_0 and a Nyquist bin are real
                    f1.y = 0.f;
                    f2.y = 0.f;
                } else if (j > mmax) {  // mirrored bin: conj
                    f1.y = -f1.y;
                    f2.y = -f2.y;
                }
                a = make_float2(f1.x - f2.y, f1.y + f2.x);
            }
        }
        A[c * n1 + r] = a;
    }
    __syncthreads();
    A = mixed_passes<DIR, kMixedThreads>(A, B, n1, C, sch, tw);
    const uint32_t lomask = (1u << lobits) - 1u;
#pragma unroll 4
    for (int idx = tid; idx < C * n1; idx += kMixedThreads) {
        const int k1 = mdiv(idx, cmagic), c = idx - k1 * C;
        if (c0 + c >= n2) continue;
        const uint32_t q = (uint32_t)(c0 + c) * (uint32_t)k1;  // < n: no reduction needed
        const float2 w = cmul(__ldg(hi + (q >> lobits)), __ldg(lo + (q & lomask)));
        stg_stream(y + (int64_t)k1 * n2 + c0 + c, ctw<DIR>(A[c * n1 + k1], w));
    }
}

// batch: transforms (real modes: (nrows + 1) / 2).
template <int MODE, int DIR>
cudaError_t launch_mixed_cols(const void* in, float2* out, int64_t batch, int n1, int n2,
                              const MixedSched& sch, const float2* tw, const float2* hi,
                              const float2* lo, int lobits, const float2* ph, int shift_in,
                              int64_t nrows, int mmax, int mmajor, cudaStream_t stream) {
    auto kern = k_mixed_cols<MODE, DIR>;
    static LaunchCache cache;
    LaunchGeom geo;
    cudaError_t e = cache.get(
        [&](int, LaunchGeom*) {
            return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)mixed_cols_smem_bytes(kMaxMixedN1));
        },
        &geo);
    if (e != cudaSuccess) return e;
    if (n1 < 2 || n1 > kMaxMixedN1 || n2 < 2) return cudaErrorInvalidValue;
    const int C = mixed_cols_per_cta(n1);
    const int64_t tiles = (n2 + C - 1) / C;
    const int64_t grid = batch * tiles;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, kMixedThreads, mixed_cols_smem_bytes(n1), stream>>>(
        in, out, n1, n2, C, div_magic((uint32_t)C), tiles, sch, tw, hi, lo, lobits, ph,
        shift_in, nrows, mmax, mmajor);
    return cudaGetLastError();
}

// The unpack after the analysis of two real rows per transform: Y = the n-point spectra
// [ntr][n] of y = x1 + i x2; bins m <= mmax of both rows, X1_m = (Y_m + conj Y_{n-m})/2,
// X2_m = (Y_m - conj Y_{n-m})/(2i) (Mota §2.6 Eq. 17-18), bins 0 and n/2 real, into the
// spectrum layout.  Grid: (m blocks, transforms).
__global__ void __launch_bounds__(kMixedThreads)
    k_mixed_unpack(const float2* __restrict__ Y, float2* F, int64_t nrows, int n, int mmax,
                   int mmajor) {
    const int64_t ntr = (nrows + 1) / 2;
    for (int64_t t = blockIdx.y; t < ntr; t += gridDim.y) {
        const float2* yr = Y + t * n;
        const int64_t r1 = 2 * t;
        const bool has2 = r1 + 1 < nrows;
        for (int m = blockIdx.x * kMixedThreads + (int)threadIdx.x; m <= mmax;
             m += gridDim.x * kMixedThreads) {
            const float2 ym = ldg_stream(yr + m), yn = ldg_stream(yr + (m == 0 ? 0 : n - m));
            float2 f1 = make_float2(0.5f * (ym.x + yn.x), 0.5f * (ym.y - yn.y));
            float2 f2 = make_float2(0.5f * (ym.y + yn.y), 0.5f * (yn.x - ym.x));
            if (m == 0 || 2 * m == n) {  // real bins: drop the rounding residue
                f1.y = 0.f;
                f2.y = 0.f;
            }
            stg_stream(F + (mmajor ? (int64_t)m * nrows + r1 : r1 * (mmax + 1) + m), f1);
            if (has2)
                stg_stream(F + (mmajor ? (int64_t)m * nrows + r1 + 1 : (r1 + 1) * (mmax + 1) + m),
                           f2);
        }
    }
}

template <int MODE, int DIR>
cudaError_t launch_mixed(const void* in, void* out, int64_t nrows, int n, const MixedSched& sch,
                         const float2* tw, const float2* ph, int shift_in, int shift_out,
                         float scale, int mmax, int mmajor, int tn1, cudaStream_t stream,
                         int64_t nreal = 0) {
    if (n < 2 || n > kMaxMixedN) return cudaErrorInvalidValue;
    const bool pair = MODE == BLU_R2C2 || MODE == BLU_C2R2;
    const int64_t ntr = pair ? (nrows + 1) / 2 : nrows;
    constexpr bool onepass = MODE != kMixedRowsT && MODE != kMixedRowsT2;
    const bool small = onepass && mixed_small_cta(n, ntr);
    auto kern = small ? k_mixed<MODE, DIR, kMixedSmallThreads> : k_mixed<MODE, DIR, kMixedThreads>;
    static LaunchCache cache;
    LaunchGeom geo;
    cudaError_t e = cache.get(
        [&](int, LaunchGeom*) {
            cudaError_t r = cudaFuncSetAttribute(k_mixed<MODE, DIR, kMixedThreads>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)mixed_smem_bytes(kMaxMixedN));
            if (r != cudaSuccess || !onepass) return r;
            return cudaFuncSetAttribute(k_mixed<MODE, DIR, kMixedSmallThreads>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)mixed_smem_bytes_for(1024, true));
        },
        &geo);
    if (e != cudaSuccess) return e;
    const int W = mixed_rows_for(n, small);
    const int64_t grid = (ntr + W - 1) / W;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, small ? kMixedSmallThreads : kMixedThreads,
           mixed_smem_bytes_for(n, small), stream>>>(
        in, out, nrows, n, W, sch, tw, ph, shift_in, shift_out, scale, mmax, mmajor,
        div_magic((uint32_t)W), div_magic((uint32_t)(mmax + 1)), tn1, nreal);
    return cudaGetLastError();
}

}  // namespace gbfft
