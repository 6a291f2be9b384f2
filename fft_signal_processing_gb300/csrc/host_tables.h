// Host construction of the twiddle tables (double precision, rounded once to float), in the
// layout the kernels read (tw_pass_off / tw_stride in fft_common.cuh).  Header-only, host code.
#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <vector>

#include "fft_common.cuh"

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

}  // namespace host
}  // namespace gbfft
