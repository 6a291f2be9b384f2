// Small transforms (N = 2^0 .. 2^4 points): one row per thread, whole DFT in registers.
//
// A CTA owns 256 consecutive rows, a contiguous block of 256*N complex64.  The block moves
// between HBM and shared memory with fully coalesced 16-byte accesses (each lane a float4, i.e.
// two points), and sits in shared memory with one padding slot per row (row stride N + 1), so
// that the 256 threads, each reading or writing its own row, hit distinct banks.  The DFT
// itself is the in-register radix-N butterfly of fft_common.cuh.
#pragma once

#include "fft_common.cuh"

namespace gbfft {

template <int LOG2N, int DIR>
__global__ void __launch_bounds__(256)
    k_small(const float2* in, float2* out, int64_t nrows, int flags, int row_parity) {
    constexpr int N = 1 << LOG2N;
    constexpr int ROWS = 256;
    constexpr int RS = N + 1;  // padded row stride in shared memory
    __shared__ float2 sm[ROWS * RS];
    const int tid = (int)threadIdx.x;
    const int64_t row0 = (int64_t)blockIdx.x * ROWS;
    const int64_t rows_here = nrows - row0 < ROWS ? nrows - row0 : ROWS;
    const int64_t pts = rows_here * N;  // points of this block (N >= 1)

    // coalesced load: point pairs (float4) when possible, the odd tail point alone
    const float2* src = in + row0 * N;
    if constexpr (N >= 2) {
        const float4* src4 = reinterpret_cast<const float4*>(src);
#pragma unroll
        for (int k = 0; k < N / 2; ++k) {
            const int i2 = tid + k * ROWS;  // float4 index in the block
            if ((int64_t)i2 * 2 < pts) {
                const float4 q = ldg_stream4(src4 + i2);
                const int p = 2 * i2, w = p >> LOG2N, e = p & (N - 1);
                sm[w * RS + e] = make_float2(q.x, q.y);
                sm[w * RS + e + 1] = make_float2(q.z, q.w);
            }
        }
    } else {
        if (tid < pts) sm[tid * RS] = ldg_stream(src + tid);
    }
    __syncthreads();

    if (tid < rows_here) {
        const int rp = row_parity ? (int)((row0 + tid) & 1) : 0;
        float2 v[N];
#pragma unroll
        for (int e = 0; e < N; ++e) {
            float2 x = sm[tid * RS + e];
            if (flags & KF_CHESS_LOAD) x = neg_if(x, (e + rp) & 1);
            v[e] = x;
        }
        dft_reg<N, DIR>(v);
#pragma unroll
        for (int k = 0; k < N; ++k) {
            float2 y = v[k];
            if (flags & KF_CHESS_STORE) y = neg_if(y, (k + rp) & 1);
            y = scale_pow2(y, flags);
            sm[tid * RS + k] = y;  // only this thread touches its row
        }
    }
    __syncthreads();

    float2* dst = out + row0 * N;
    if constexpr (N >= 2) {
        float4* dst4 = reinterpret_cast<float4*>(dst);
#pragma unroll
        for (int k = 0; k < N / 2; ++k) {
            const int i2 = tid + k * ROWS;
            if ((int64_t)i2 * 2 < pts) {
                const int p = 2 * i2, w = p >> LOG2N, e = p & (N - 1);
                const float2 a = sm[w * RS + e], b = sm[w * RS + e + 1];
                stg_stream4(dst4 + i2, make_float4(a.x, a.y, b.x, b.y));
            }
        }
    } else {
        if (tid < pts) stg_stream(dst + tid, sm[tid * RS]);
    }
}

template <int LOG2N, int DIR>
cudaError_t launch_small(const float2* in, float2* out, int64_t nrows, int flags, int row_parity,
                         cudaStream_t stream) {
    const int64_t grid = (nrows + 255) / 256;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    k_small<LOG2N, DIR><<<(unsigned)grid, 256, 0, stream>>>(in, out, nrows, flags, row_parity);
    return cudaGetLastError();
}

}  // namespace gbfft
