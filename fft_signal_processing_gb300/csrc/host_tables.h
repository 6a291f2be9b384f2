// Host construction of the twiddle tables (double precision, rounded once to float), in the
// layout the kernels read (tw_pass_off / tw_stride in fft_common.cuh).  Header-only, host code.
#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <complex>
#include <cstdint>
#include <cstdlib>
#include <vector>

#include "fft_common.cuh"
#include "kernels.h"

namespace gbfft {
namespace host {

// (cos, sin)(2*pi*q/m) in double, rounded once to float.  The angle is reduced in integers to
// the first quadrant, and cos/sin are evaluated at the nearer of a and pi/2 - a, so quarter
// turns are exactly 0 and +-1 and the table keeps the symmetries of the unit circle.
inline float2 root_of_unity(int64_t q, int64_t m) {
    const double two_pi = 6.283185307179586476925286766559005768;
    q %= m;
    if (q < 0) q += m;
    if (m % 4 != 0) return make_float2(2 * q == m ? -1.f : 1.f, 0.f);  // m = 1, 2
    const int64_t qq = m / 4, quad = q / qq, a = q % qq;
    double c, s;
    if (a == 0) {
        c = 1.0;
        s = 0.0;
    } else if (a <= qq / 2) {
        c = std::cos(two_pi * (double)a / (double)m);
        s = std::sin(two_pi * (double)a / (double)m);
    } else {  // complementary angle pi/2 - th for accuracy near pi/2
        c = std::sin(two_pi * (double)(qq - a) / (double)m);
        s = std::cos(two_pi * (double)(qq - a) / (double)m);
    }
    double x, y;  // rotate by quad quarter turns
    switch (quad & 3) {
        case 0: x = c; y = s; break;
        case 1: x = -s; y = c; break;
        case 2: x = -c; y = -s; break;
        default: x = s; y = -c; break;
    }
    return make_float2((float)x, (float)y);
}

// (cos, sin)(2*pi*q/m) for any m >= 1: the power-of-two moduli through root_of_unity; others
// with q reduced modulo m in integers and the angle folded to [0, pi] (sin changes sign), in
// double precision rounded once to float.
inline float2 root_any(int64_t q, int64_t m) {
    q %= m;
    if (q < 0) q += m;
    if ((m & (m - 1)) == 0) return root_of_unity(q, m);
    const double two_pi = 6.283185307179586476925286766559005768;
    const bool upper = 2 * q > m;
    const int64_t a = upper ? m - q : q;
    const double th = two_pi * (double)a / (double)m;
    const double s = std::sin(th);
    return make_float2((float)std::cos(th), (float)(upper ? -s : s));
}

inline void align_table(std::vector<float2>& v) {
    while (v.size() % 32) v.push_back(make_float2(0.f, 0.f));
}

// Per-pass tables of a 2^l-point transform with largest radix 2^maxrb; returns the offset.
inline size_t append_pass_tables(std::vector<float2>& v, int l, int maxrb) {
    align_table(v);
    const size_t off = v.size();
    const int npass = sched_npass(l, maxrb);
    for (int p = 1; p < npass; ++p) {
        const int rb = sched_rbits(l, maxrb, p);
        const int64_t R = int64_t(1) << rb, Ns = int64_t(1) << sched_span_bits(l, maxrb, p);
        const int A = tw_lo_count(rb), B = tw_hi_count(rb), S = tw_stride(rb);
        for (int64_t m = 0; m < Ns; ++m) {
            for (int a = 0; a < A; ++a) v.push_back(root_of_unity(m * a, Ns * R));
            for (int b = 0; b < B; ++b) v.push_back(root_of_unity(m * A * b, Ns * R));
            for (int k = A + B; k < S; ++k) v.push_back(make_float2(0.f, 0.f));
        }
    }
    if (v.size() - off != (size_t)tw_table_size(l, maxrb)) std::abort();  // layout invariant
    return off;
}

// w_m^(q*step) for q < count; returns the offset.
inline size_t append_roots(std::vector<float2>& v, int64_t count, int64_t step, int64_t m) {
    align_table(v);
    const size_t off = v.size();
    for (int64_t q = 0; q < count; ++q) v.push_back(root_of_unity(q * step, m));
    return off;
}

// ---- mixed-radix schedule tables ----------------------------------------------------------
// Pass p of radix R and span Ns: (cos, sin)(2*pi*m*r/(Ns*R)) at m*(R-1) + r-1, m < Ns,
// 1 <= r < R.  Fills sch (spans, radices, offsets relative to the returned offset).
inline size_t append_mixed_tables(std::vector<float2>& v, int npass, const int* radix,
                                  MixedSched* sch) {
    align_table(v);
    const size_t off = v.size();
    sch->npass = npass;
    int64_t ns = 1;
    for (int p = 0; p < npass; ++p) {
        const int R = radix[p];
        sch->radix[p] = R;
        sch->span[p] = (int)ns;
        sch->smagic[p] = div_magic((uint32_t)ns);
        sch->off[p] = (int)(v.size() - off);
        for (int64_t m = 0; m < ns; ++m)
            for (int r = 1; r < R; ++r) v.push_back(root_any(m * r, ns * R));
        ns *= R;
    }
    for (int p = 0; p < npass; ++p) sch->qmagic[p] = div_magic((uint32_t)(ns / radix[p]));
    sch->nmagic = div_magic((uint32_t)ns);
    return off;
}

// (cos, sin)(2*pi*q*step/m) for q < count, any m; returns the offset.
inline size_t append_roots_any(std::vector<float2>& v, int64_t count, int64_t step, int64_t m) {
    align_table(v);
    const size_t off = v.size();
    for (int64_t q = 0; q < count; ++q)
        v.push_back(root_any((int64_t)(((__int128)q * step) % m), m));
    return off;
}

// (cos, sin)(2*pi*(j*h mod n)/n) for j < n: the fftshift phase of a length-n row.
inline size_t append_phase(std::vector<float2>& v, int64_t n, int64_t h) {
    align_table(v);
    const size_t off = v.size();
    for (int64_t j = 0; j < n; ++j) v.push_back(root_any((int64_t)(((__int128)j * h) % n), n));
    return off;
}

// ---- chirp-z (Bluestein) tables for a length-n transform of sign s, n not a power of two ----
// With j*k = (j^2 + k^2 - (k-j)^2) / 2 the DFT becomes a convolution:
//   X_k = c_k * sum_j (x_j c_j) b_{k-j},   c_j = exp(s*pi*i*j^2/n),   b_d = conj(c_d),
// evaluated with m-point FFTs (m a power of two, m >= 2n-1, so the circular convolution of
// the zero-padded sequences equals the linear one on k < n).  j^2 is reduced modulo 2n in
// integers before the angle is formed.

inline std::complex<double> chirp(int64_t j, int64_t n, int sign) {
    const double pi = 3.141592653589793238462643383279502884;
    const int64_t q = (int64_t)(((unsigned __int128)(j < 0 ? -j : j) * (uint64_t)(j < 0 ? -j : j)) %
                                (uint64_t)(2 * n));
    const double th = pi * (double)q / (double)n;
    return {std::cos(th), (double)sign * std::sin(th)};
}

// In-place iterative radix-2 FFT in double precision (sign s, unnormalised), a.size() a power
// of two; each twiddle is evaluated directly (no recurrence).  Plan-time use only.
inline void fft_fp64(std::vector<std::complex<double>>& a, int sign) {
    const size_t m = a.size();
    for (size_t i = 1, j = 0; i < m; ++i) {  // bit-reversal permutation
        size_t bit = m >> 1;
        for (; j & bit; bit >>= 1) j ^= bit;
        j ^= bit;
        if (i < j) std::swap(a[i], a[j]);
    }
    const double two_pi = 6.283185307179586476925286766559005768;
    for (size_t len = 2; len <= m; len <<= 1) {
        for (size_t k = 0; k < len / 2; ++k) {
            const double th = two_pi * (double)k / (double)len;
            const std::complex<double> w(std::cos(th), (double)sign * std::sin(th));
            for (size_t i = 0; i < m; i += len) {
                const std::complex<double> u = a[i + k], t = w * a[i + k + len / 2];
                a[i + k] = u + t;
                a[i + k + len / 2] = u - t;
            }
        }
    }
}

// c_j * exp(2*pi*i*j*q/n) for j < n (q = 0: the plain chirp; q = +-floor(n/2): the chirp with
// the fftshift folded in, see append_chirp's callers); the two angles are reduced in integers
// and added in double precision before one cos/sin.  Returns the offset.
inline size_t append_chirp(std::vector<float2>& v, int64_t n, int sign, int64_t q = 0) {
    const double pi = 3.141592653589793238462643383279502884;
    align_table(v);
    const size_t off = v.size();
    for (int64_t j = 0; j < n; ++j) {
        const int64_t a = (int64_t)(((unsigned __int128)j * (uint64_t)j) % (uint64_t)(2 * n));
        int64_t b = (int64_t)(((__int128)j * q) % n);
        if (b < 0) b += n;
        const double th = (double)sign * pi * (double)a / (double)n + 2.0 * pi * (double)b / (double)n;
        v.push_back(make_float2((float)std::cos(th), (float)std::sin(th)));
    }
    return off;
}

// FFT_m^(-)(b) / m with b_d = conj(c_d) placed circularly (d and m - d for |d| < n); returns
// the offset.
inline size_t append_chirp_filter(std::vector<float2>& v, int64_t n, int64_t m, int sign) {
    std::vector<std::complex<double>> b((size_t)m, std::complex<double>(0.0, 0.0));
    for (int64_t d = 0; d < n; ++d) {
        const std::complex<double> c = std::conj(chirp(d, n, sign));
        b[(size_t)d] = c;
        if (d > 0) b[(size_t)(m - d)] = c;
    }
    fft_fp64(b, -1);
    align_table(v);
    const size_t off = v.size();
    for (int64_t q = 0; q < m; ++q)
        v.push_back(make_float2((float)(b[(size_t)q].real() / (double)m),
                                (float)(b[(size_t)q].imag() / (double)m)));
    return off;
}

}  // namespace host
}  // namespace gbfft
