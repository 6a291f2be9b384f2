// Band-limited real rows, two rows per complex transform (Mota, "High Performance Fourier
// Transforms on GPUs with GLSL", §2.6 Eq. 17-18, "two real inputs within one complex").
//
// Rows x1 = row 2p and x2 = row 2p+1 (N = 2^LOG2N real points each) are packed as the complex
// row y = x1 + i x2, and one N-point complex FFT serves both.  With Y = FFT_N(y) and
// Y_N = Y_0, the spectra of the two real rows are
//     X1_k = (Y_k + conj Y_{N-k}) / 2,      X2_k = (Y_k - conj Y_{N-k}) / (2i)
// (the unpacking of Eq. 18, whose printed form is garbled: this is the form that follows from
// the Hermitian symmetry X_{N-k} = conj X_k of a real row's spectrum).  Synthesis runs the same
// identity backwards: Y_k = X1_k + i X2_k over the Hermitian-extended spectra
// (X_0 = Re F_0, X_m = F_m and X_{N-m} = conj F_m for 1 <= m <= mmax, other bins 0, a Nyquist
// bin m = N/2 real), y = inverse FFT_N(Y) unnormalised, x1 = Re y, x2 = Im y.  The band-limited
// analysis and synthesis are those of "src/sht/wgsl/fourier.ts" (header comment).
//
// One CTA holds W row pairs; a pair's threads are adjacent lanes, so the real rows are read and
// written with coalesced 4-byte accesses.  The spectrum side goes through shared memory: the
// unpack needs Y_k and Y_{N-k} together, and the gather builds Y_k and Y_{N-k} from one read
// of F1_m and F2_m.  An odd row count pairs the last row with a zero row that is never stored.
#pragma once

#include "fft_kernel.cuh"

namespace gbfft {

template <class C>
struct RealPairCfg {
    static_assert(C::TFAST, "a pair's threads are adjacent lanes (coalesced row accesses)");
    static constexpr int SLOTS = C::SROW > C::N ? C::SROW : C::N;  // per pair: exchange or Y
    static constexpr size_t SMEM_BYTES = (size_t)SLOTS * C::W * sizeof(float2);
};

// R2C: in = real rows [nrows][N] float32; out = spectrum rows [nrows][mmax+1] (row-major) or
// [mmax+1][nrows] (m-major), 0 <= mmax <= N/2.  IDX: the index-only diagnostic (no core
// transform: Y = y, so the pack, the unpack and the layout are exercised alone).
template <class C, bool IDX = false>
__global__ void __launch_bounds__(C::THREADS)
    k_r2c_pair(const float* in, float2* out, int64_t nrows, int mmax, int mmajor,
               const float2* __restrict__ tw) {
    constexpr int N = C::N;
    constexpr int W = C::W;
    constexpr int SLOTS = RealPairCfg<C>::SLOTS;
    extern __shared__ __align__(16) float2 smem[];
    const int w = (int)threadIdx.x / C::T;
    const int t = (int)threadIdx.x % C::T;
    const int64_t npairs = (nrows + 1) / 2;
    const int64_t p0 = (int64_t)blockIdx.x * W;
    const int64_t pr = p0 + w;
    const bool a1 = pr < npairs, a2 = 2 * pr + 1 < nrows;
    float2* sb = smem + w * SLOTS;

    constexpr int R0 = C::radix(0);
    constexpr int B0 = C::E / R0;
    constexpr int S0 = C::N / R0;
    const float* x1 = in + (a1 ? 2 * pr * N : 0);
    const float* x2 = in + (a2 ? (2 * pr + 1) * N : 0);
    float2 v[C::E];
#pragma unroll
    for (int b = 0; b < B0; ++b) {
        const int j = t + b * C::T;
#pragma unroll
        for (int r = 0; r < R0; ++r) {
            const int e = j + r * S0;
            v[b * R0 + r] = make_float2(a1 ? __ldcs(x1 + e) : 0.f, a2 ? __ldcs(x2 + e) : 0.f);
        }
    }
    if constexpr (IDX)
        identity_passes<C>(v, t, sb);
    else
        run_passes<C, -1, 0>(v, t, sb, tw);

    constexpr int RL = C::radix(C::NPASS - 1);
    constexpr int BL = C::E / RL;
    constexpr int SL = C::N / RL;
    if constexpr (C::NPASS > 1) __syncthreads();  // the last exchange has been read
#pragma unroll
    for (int b = 0; b < BL; ++b) {
        const int j = t + b * C::T;
#pragma unroll
        for (int r = 0; r < RL; ++r) sb[j + r * SL] = v[b * RL + r];  // Y_k, dense
    }
    __syncthreads();

    const int nm = mmax + 1;
    const int total = W * nm;
    for (int i = (int)threadIdx.x; i < total; i += C::THREADS) {
        // m-major: the W pairs are adjacent lanes (consecutive spectrum rows); row-major:
        // consecutive bins m of one pair are
        const int w2 = mmajor ? i % W : i / nm;
        const int m = mmajor ? i / W : i % nm;
        const int64_t p = p0 + w2;
        if (p >= npairs) continue;
        const float2 ym = smem[w2 * SLOTS + m];
        const float2 yn = smem[w2 * SLOTS + ((N - m) & (N - 1))];
        const float2 f1 = make_float2(0.5f * (ym.x + yn.x), 0.5f * (ym.y - yn.y));
        const float2 f2 = make_float2(0.5f * (ym.y + yn.y), 0.5f * (yn.x - ym.x));
        const int64_t r1 = 2 * p;
        const bool has2 = r1 + 1 < nrows;
        if (mmajor) {
            float2* o = out + (int64_t)m * nrows + r1;
            if (has2 && (((uintptr_t)o & 15u) == 0)) {
                stg_stream4(reinterpret_cast<float4*>(o), make_float4(f1.x, f1.y, f2.x, f2.y));
            } else {
                stg_stream(o, f1);
                if (has2) stg_stream(o + 1, f2);
            }
        } else {
            stg_stream(out + r1 * nm + m, f1);
            if (has2) stg_stream(out + (r1 + 1) * nm + m, f2);
        }
    }
}

// C2R: in = spectrum (layout as above); out = real rows [nrows][N] float32.  IDX: the
// index-only diagnostic (no core transform: x1 = Re Y, x2 = Im Y of the assembled Y).
template <class C, bool IDX = false>
__global__ void __launch_bounds__(C::THREADS)
    k_c2r_pair(const float2* in, float* out, int64_t nrows, int mmax, int mmajor,
               const float2* __restrict__ tw) {
    constexpr int N = C::N;
    constexpr int W = C::W;
    constexpr int SLOTS = RealPairCfg<C>::SLOTS;
    constexpr int H = N / 2;
    extern __shared__ __align__(16) float2 smem[];
    const int w = (int)threadIdx.x / C::T;
    const int t = (int)threadIdx.x % C::T;
    const int64_t npairs = (nrows + 1) / 2;
    const int64_t p0 = (int64_t)blockIdx.x * W;
    const int64_t pr = p0 + w;
    float2* sb = smem + w * SLOTS;
    const int nm = mmax + 1;

    // Y_m and Y_{N-m} from one read of F1_m, F2_m (m = 0..N/2), zero above mmax
    const int total = W * (H + 1);
    for (int i = (int)threadIdx.x; i < total; i += C::THREADS) {
        const int w2 = mmajor ? i % W : i / (H + 1);
        const int m = mmajor ? i / W : i % (H + 1);
        const int64_t p = p0 + w2;
        const int64_t r1 = 2 * p;
        float2 f1 = make_float2(0.f, 0.f), f2 = make_float2(0.f, 0.f);
        if (p < npairs && m <= mmax) {
            const bool has2 = r1 + 1 < nrows;
            if (mmajor) {
                const float2* s = in + (int64_t)m * nrows + r1;
                if (has2 && (((uintptr_t)s & 15u) == 0)) {
                    const float4 q = ldg_stream4(reinterpret_cast<const float4*>(s));
                    f1 = make_float2(q.x, q.y);
                    f2 = make_float2(q.z, q.w);
                } else {
                    f1 = ldg_stream(s);
                    if (has2) f2 = ldg_stream(s + 1);
                }
            } else {
                f1 = ldg_stream(in + r1 * nm + m);
                if (has2) f2 = ldg_stream(in + (r1 + 1) * nm + m);
            }
            if (m == 0 || m == H) {  // X_0 and the Nyquist bin are real
                f1.y = 0.f;
                f2.y = 0.f;
            }
        }
        // Y_m = X1_m + i X2_m; Y_{N-m} = conj X1_m + i conj X2_m
        smem[w2 * SLOTS + m] = make_float2(f1.x - f2.y, f1.y + f2.x);
        if (m != 0 && m != H) smem[w2 * SLOTS + (N - m)] = make_float2(f1.x + f2.y, f2.x - f1.y);
    }
    __syncthreads();

    constexpr int R0 = C::radix(0);
    constexpr int B0 = C::E / R0;
    constexpr int S0 = C::N / R0;
    float2 v[C::E];
#pragma unroll
    for (int b = 0; b < B0; ++b) {
        const int j = t + b * C::T;
#pragma unroll
        for (int r = 0; r < R0; ++r) v[b * R0 + r] = sb[j + r * S0];
    }
    if constexpr (C::NPASS > 1) __syncthreads();  // the buffer becomes the exchange buffer
    if constexpr (IDX)
        identity_passes<C>(v, t, sb);
    else
        run_passes<C, +1, 0>(v, t, sb, tw);

    constexpr int RL = C::radix(C::NPASS - 1);
    constexpr int BL = C::E / RL;
    constexpr int SL = C::N / RL;
    if (pr < npairs) {
        const bool has2 = 2 * pr + 1 < nrows;
        float* x1 = out + 2 * pr * N;
        float* x2 = x1 + N;
#pragma unroll
        for (int b = 0; b < BL; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < RL; ++r) {
                const int k = j + r * SL;
                __stcs(x1 + k, v[b * RL + r].x);
                if (has2) __stcs(x2 + k, v[b * RL + r].y);
            }
        }
    }
}

template <class C, bool IDX>
cudaError_t launch_real_pair_impl(bool analysis, const void* in, void* out, int64_t nrows,
                                  int mmax, int mmajor, const float2* tw, cudaStream_t stream) {
    constexpr size_t smem = RealPairCfg<C>::SMEM_BYTES;
    const int64_t npairs = (nrows + 1) / 2;
    const int64_t grid = (npairs + C::W - 1) / C::W;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (analysis) {
        auto kern = k_r2c_pair<C, IDX>;
        static LaunchCache cache;
        LaunchGeom geo;
        cudaError_t e = cache.get(
            [&](int, LaunchGeom*) {
                return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)smem);
            },
            &geo);
        if (e != cudaSuccess) return e;
        kern<<<(unsigned)grid, C::THREADS, smem, stream>>>(static_cast<const float*>(in),
                                                           static_cast<float2*>(out), nrows,
                                                           mmax, mmajor, tw);
    } else {
        auto kern = k_c2r_pair<C, IDX>;
        static LaunchCache cache;
        LaunchGeom geo;
        cudaError_t e = cache.get(
            [&](int, LaunchGeom*) {
                return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            (int)smem);
            },
            &geo);
        if (e != cudaSuccess) return e;
        kern<<<(unsigned)grid, C::THREADS, smem, stream>>>(static_cast<const float2*>(in),
                                                           static_cast<float*>(out), nrows,
                                                           mmax, mmajor, tw);
    }
    return cudaGetLastError();
}

// The index-only diagnostic (KF_INDEX_ONLY in flags) is instantiated for 4096-point rows only.
template <class C>
cudaError_t launch_real_pair(bool analysis, const void* in, void* out, int64_t nrows, int mmax,
                             int mmajor, const float2* tw, int flags, cudaStream_t stream) {
    if (flags & KF_INDEX_ONLY) {
        if constexpr (C::LOG2N == 12)
            return launch_real_pair_impl<C, true>(analysis, in, out, nrows, mmax, mmajor, tw,
                                                  stream);
        else
            return cudaErrorNotSupported;
    }
    return launch_real_pair_impl<C, false>(analysis, in, out, nrows, mmax, mmajor, tw, stream);
}

}  // namespace gbfft
