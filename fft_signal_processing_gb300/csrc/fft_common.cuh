// Device building blocks shared by every kernel of the library: complex arithmetic on
// float2 (x = re, y = im), twiddle multiplication, the in-register radix-R butterflies and the
// shared-memory padding used by the exchanges between radix passes.
//
// Convention: DIR is the sign s of the exponent, -1 forward, +1 inverse (Mota, "High
// Performance Fourier Transforms on GPUs with GLSL", §2.2 Eq. 5 and §2.3.1 Algorithm 2:
// the inverse is the same algorithm with exp(+2*pi*i/m)).  Twiddle tables always store
// (cos t, sin t) for t >= 0; the sign is applied at use, as the WGSL Stockham kernels of
// "src/sht/wgsl/fourier.ts" do with their (cos, sin) table.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace gbfft {

__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
__device__ __forceinline__ float2 cneg(float2 a) { return make_float2(-a.x, -a.y); }

// a * exp(DIR * i * t) given w = (cos t, sin t).
template <int DIR>
__device__ __forceinline__ float2 ctw(float2 a, float2 w) {
    if constexpr (DIR < 0)
        return make_float2(fmaf(a.x, w.x, a.y * w.y), fmaf(a.y, w.x, -(a.x * w.y)));
    else
        return make_float2(fmaf(a.x, w.x, -(a.y * w.y)), fmaf(a.x, w.y, a.y * w.x));
}

// Plain complex product a*b.
__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
    return make_float2(fmaf(a.x, b.x, -(a.y * b.y)), fmaf(a.x, b.y, a.y * b.x));
}

// cos(2*pi*k/64) for any integer k, as compile-time constants (quarter-wave values of the
// 64th roots of unity; every in-register butterfly radix used here divides 64).
__host__ __device__ constexpr double cos64(int k) {
    k = ((k % 64) + 64) % 64;
    if (k > 32) k = 64 - k;          // cos is even
    const bool neg = k > 16;         // cos(pi - a) = -cos(a)
    if (neg) k = 32 - k;
    double v = 0.0;
    switch (k) {
        case 0: v = 1.0; break;
        case 1: v = 0.99518472667219688624483695310948; break;
        case 2: v = 0.98078528040323044912618223613424; break;
        case 3: v = 0.95694033573220886493579788698027; break;
        case 4: v = 0.92387953251128675612818318939679; break;
        case 5: v = 0.88192126434835502971275686366039; break;
        case 6: v = 0.83146961230254523707878837761791; break;
        case 7: v = 0.77301045336273696081090660975847; break;
        case 8: v = 0.70710678118654752440084436210485; break;
        case 9: v = 0.63439328416364549821517161322549; break;
        case 10: v = 0.55557023301960222474283081394853; break;
        case 11: v = 0.47139673682599764855638762591373; break;
        case 12: v = 0.38268343236508977172845998403040; break;
        case 13: v = 0.29028467725446236763619237581740; break;
        case 14: v = 0.19509032201612826784828486847702; break;
        case 15: v = 0.09801714032956060199419556388864; break;
        default: v = 0.0; break;
    }
    return neg ? -v : v;
}
__host__ __device__ constexpr double sin64(int k) { return cos64(k - 16); }

// a * exp(DIR * 2*pi*i * E / R) with E, R compile-time.  Quarter turns are exact swaps and
// sign flips; everything else is one complex multiply by float constants.
template <int DIR, int E, int R>
__device__ __forceinline__ float2 crot(float2 a) {
    constexpr int e = ((E % R) + R) % R;
    if constexpr (e == 0) {
        return a;
    } else if constexpr (4 * e == R) {          // DIR * i
        return DIR < 0 ? make_float2(a.y, -a.x) : make_float2(-a.y, a.x);
    } else if constexpr (2 * e == R) {          // -1
        return cneg(a);
    } else if constexpr (4 * e == 3 * R) {      // -DIR * i
        return DIR < 0 ? make_float2(-a.y, a.x) : make_float2(a.y, -a.x);
    } else {
        static_assert(64 % R == 0, "radix must divide 64");
        constexpr int k = e * (64 / R);
        constexpr float c = (float)cos64(k);
        constexpr float s = (float)(DIR * sin64(k));
        return make_float2(fmaf(a.x, c, -(a.y * s)), fmaf(a.x, s, a.y * c));
    }
}

__host__ __device__ constexpr int ilog2c(int v) { return v <= 1 ? 0 : 1 + ilog2c(v >> 1); }

// ---- pass schedule ----------------------------------------------------------------------------
// A 2^l-point transform is split into npass radix passes of at most 2^m points each, as evenly
// as possible with the larger radices first (e.g. l = 12, m = 6: 64 x 64; l = 10, m = 4:
// 16 x 8 x 8).  Shared by the kernels and the host twiddle-table builder.
__host__ __device__ constexpr int sched_npass(int l, int m) { return l <= 0 ? 1 : (l + m - 1) / m; }
__host__ __device__ constexpr int sched_rbits(int l, int m, int p) {
    return l / sched_npass(l, m) + (p < l % sched_npass(l, m) ? 1 : 0);
}
__host__ __device__ constexpr int sched_span_bits(int l, int m, int p) {
    return p <= 0 ? 0 : sched_span_bits(l, m, p - 1) + sched_rbits(l, m, p - 1);
}

// ---- twiddle tables ---------------------------------------------------------------------------
// Pass p >= 1 (radix R = 2^rb, span Ns) multiplies element r of butterfly j by w^r, where
// w = w_{Ns*R}^(j mod Ns).  Its table holds, for each m < Ns, the A = 2^ceil(rb/2) "low"
// powers w^a (a < A) followed by the B = R/A "high" powers w^(A*b) (b < B), padded to an even
// count; w^r with r = a + A*b is formed as w^a * w^(A*b).  Passes are stored back to back.
__host__ __device__ constexpr int tw_lo_count(int rb) { return 1 << ((rb + 1) / 2); }
__host__ __device__ constexpr int tw_hi_count(int rb) { return 1 << (rb - (rb + 1) / 2); }
__host__ __device__ constexpr int tw_stride(int rb) {
    return ((tw_lo_count(rb) + tw_hi_count(rb)) + 1) & ~1;
}
__host__ __device__ constexpr int tw_pass_off(int l, int m, int p) {
    return p <= 1 ? 0
                  : tw_pass_off(l, m, p - 1) +
                        (1 << sched_span_bits(l, m, p - 1)) * tw_stride(sched_rbits(l, m, p - 1));
}
__host__ __device__ constexpr int tw_table_size(int l, int m) {
    return tw_pass_off(l, m, sched_npass(l, m));
}

__host__ __device__ constexpr int bitrev_c(int i, int bits) {
    int r = 0;
    for (int b = 0; b < bits; ++b) r |= ((i >> b) & 1) << (bits - 1 - b);
    return r;
}

// In-register R-point DFT, unnormalised, sign DIR, natural order in and out:
// v[k] <- sum_j v[j] exp(DIR*2*pi*i*j*k/R).  Decimation in frequency over the register array
// (every index is a compile-time constant after unrolling, so the closing bit-reversal is only
// a renaming of registers).  Stages go two bits at a time as radix-4 butterflies, with one
// twiddle-free radix-2 stage last when log2 R is odd.  A radix-4 DIF butterfly on
// a_n = v[k + n*q] (k < q, block of 4q) writes
//   v[k]      = Y0,            v[k + q]  = Y2 * w^{2k},
//   v[k + 2q] = Y1 * w^{k},    v[k + 3q] = Y3 * w^{3k},       w = exp(DIR*2*pi*i/(4q)),
// Y_m = sum_n a_n (DIR*i)^{n*m}: exactly the positions two radix-2 DIF stages give, with one
// complex multiplication fewer.
template <int DIR, int R, int Q, int K>
__device__ __forceinline__ void dif4_bfly(float2* v) {
    const float2 a0 = v[K], a1 = v[K + Q], a2 = v[K + 2 * Q], a3 = v[K + 3 * Q];
    const float2 t0 = cadd(a0, a2), t1 = csub(a0, a2), t2 = cadd(a1, a3);
    const float2 d = csub(a1, a3);
    const float2 t3 = DIR < 0 ? make_float2(d.y, -d.x) : make_float2(-d.y, d.x);  // DIR*i*d
    constexpr int U = R / (4 * Q);  // w = exp(DIR*2*pi*i*U/R)
    v[K] = cadd(t0, t2);
    v[K + Q] = crot<DIR, 2 * K * U, R>(csub(t0, t2));
    v[K + 2 * Q] = crot<DIR, K * U, R>(cadd(t1, t3));
    v[K + 3 * Q] = crot<DIR, 3 * K * U, R>(csub(t1, t3));
}
template <int DIR, int R, int Q, int K = 0>
__device__ __forceinline__ void dif4_block(float2* v) {
    if constexpr (K < Q) {
        dif4_bfly<DIR, R, Q, K>(v);
        dif4_block<DIR, R, Q, K + 1>(v);
    }
}
// stages covering bits S.. of the index (radix-2 stage s has half-size R >> (s+1))
template <int DIR, int R, int S, int L>
__device__ __forceinline__ void dif_stages(float2* v) {
    if constexpr (S + 2 <= L) {
        constexpr int Q = R >> (S + 2);
#pragma unroll
        for (int blk = 0; blk < R; blk += 4 * Q) dif4_block<DIR, R, Q>(v + blk);
        dif_stages<DIR, R, S + 2, L>(v);
    } else if constexpr (S + 1 == L) {  // radix 2 with half-size 1: no twiddles
#pragma unroll
        for (int blk = 0; blk < R; blk += 2) {
            const float2 a = v[blk], b = v[blk + 1];
            v[blk] = cadd(a, b);
            v[blk + 1] = csub(a, b);
        }
    }
}
template <int R, int DIR>
__device__ __forceinline__ void dft_reg(float2* v) {
    constexpr int L = ilog2c(R);
    dif_stages<DIR, R, 0, L>(v);
    float2 t[R];
#pragma unroll
    for (int i = 0; i < R; ++i) t[i] = v[bitrev_c(i, L)];
#pragma unroll
    for (int i = 0; i < R; ++i) v[i] = t[i];
}

// Shared-memory index padding: one float2 of padding every 2^LP slots.  With 2^LP equal to the
// radix R0 of the first pass, the stride-R0 writes of that pass are bank-conflict free for
// 64-bit accesses, and the unit-stride accesses of the other passes stay (nearly) so.
template <int LP>
__device__ __forceinline__ int spad(int i) { return i + (i >> LP); }
__host__ __device__ constexpr int spad_size(int n, int lp) { return n + (n >> lp); }

// Streaming global loads / stores (data is touched once per pass).
__device__ __forceinline__ float2 ldg_stream(const float2* p) { return __ldcs(p); }
__device__ __forceinline__ void stg_stream(float2* p, float2 v) { __stcs(p, v); }
__device__ __forceinline__ float4 ldg_stream4(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ void stg_stream4(float4* p, float4 v) { __stcs(p, v); }

// Flags understood by the transform kernels.
enum : int {
    KF_CHESS_LOAD = 1,   // multiply input element (row, j) by (-1)^j before the transform
    KF_CHESS_STORE = 2,  // multiply output element (row, k) by (-1)^k after the transform
    KF_CHESS_ROW = 4,    // 2-D chessboard: also multiply by (-1)^row
    KF_SCALE_SHIFT = 8,  // bits 8..15 hold k: the stored output is multiplied by 2^-k (k = 0: not)
    KF_INDEX_ONLY = 16,  // diagnostic: no butterflies, twiddles or recombination (identity_passes)
};

// Flag bits asking the final store of a transform of 2^k points to scale by 1/2^k.
__host__ __device__ constexpr int kf_scale(int k) { return k << KF_SCALE_SHIFT; }

__device__ __forceinline__ float2 neg_if(float2 v, int odd) { return odd ? cneg(v) : v; }

// v * 2^-k for the k held in flags: an exact power-of-two scaling (k < 127 keeps 2^-k normal).
__device__ __forceinline__ float2 scale_pow2(float2 v, int flags) {
    const int k = (flags >> KF_SCALE_SHIFT) & 0xff;
    if (k == 0) return v;
    const float s = __int_as_float((127 - k) << 23);
    return make_float2(v.x * s, v.y * s);
}

}  // namespace gbfft
