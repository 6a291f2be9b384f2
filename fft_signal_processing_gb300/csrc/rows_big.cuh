// Persistent one-pass kernel for long rows (2^13 and 2^14 points).
//
// A row this long fills a large part of the register file, so few rows fit on an SM at once.
// To keep HBM busy anyway, each CTA holds a full-row shared-memory stage for the asynchronous
// bulk copy of the NEXT row, separate from the exchange buffer of the row being transformed:
// as soon as the current row has been read from the stage into registers, the stage is
// refilled, and the copy overlaps the whole transform.  The exchange buffer holds only half a
// row: every exchange runs in two phases.  In the Stockham ordering the destination half of
// an exchange write depends only on the butterfly index j (the top index bit is that of
// j div Ns), and the source half of a read depends only on the element r of the next pass
// (index j + r*N/R), so in phase h the butterflies writing into half h write, and every thread
// reads its elements with r in half h.
#pragma once

#include "fft_kernel.cuh"
#include "tma.cuh"

namespace gbfft {

template <int LOG2N_, int MAXRB_, int MIN_CTAS_ = 1>
struct RowsBigCfg {
    using C = FftCfg<LOG2N_, MAXRB_, 0, true>;
    static constexpr int MIN_CTAS = MIN_CTAS_;  // CTAs per SM the registers must allow
    static constexpr int N = C::N;
    static constexpr int HALF = spad_size(N / 2, C::LP);  // padded half-row exchange slots
    static constexpr size_t STAGE_BYTES = (size_t)N * sizeof(float2);
    static constexpr size_t SMEM_BYTES = STAGE_BYTES + (size_t)HALF * sizeof(float2);
    static_assert(C::NPASS >= 2, "long rows take several passes");
    static_assert(STAGE_BYTES % 128 == 0, "the exchange buffer stays 128-byte aligned");
};

// Passes P..NPASS-1 with two-phase exchanges through a half-length exchange buffer.  sb points
// at this transform's first slot; slots are C::SS apart (1 for a single row, W when W
// transforms are interleaved lane by lane).
template <class C, int DIR, int P>
__device__ __forceinline__ void run_passes_split(float2 (&v)[C::E], int t, float2* sb,
                                                 const float2* __restrict__ tw) {
    constexpr int R = C::radix(P);
    constexpr int B = C::E / R;
    constexpr int Ns = C::span(P);
    constexpr int HN = C::N / 2;
#pragma unroll
    for (int b = 0; b < B; ++b) dft_reg<R, DIR>(v + b * R);
    if constexpr (P + 1 < C::NPASS) {
        constexpr int R2 = C::radix(P + 1);
        constexpr int B2 = C::E / R2;
        constexpr int S2 = C::N / R2;
        PassTw<C, P + 1> pt[B2];
#pragma unroll
        for (int b = 0; b < B2; ++b) load_twiddles<C, P + 1>(pt[b], t + b * C::T, tw);
        // phase 0 reads (r < R2/2) wait in lo until the phase-1 writes have left v
        float2 lo[B2][R2 / 2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            __syncthreads();  // the buffer is free (previous phase or exchange fully read)
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int j = t + b * C::T;
                const int base = (j / Ns) * Ns * R + (j & (Ns - 1));
                if ((base >= HN) == (h == 1)) {  // all R outputs of j land in half h
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        sb[spad<C::LP>(base + r * Ns - h * HN) * C::SS] = v[b * R + r];
                }
            }
            __syncthreads();
#pragma unroll
            for (int b = 0; b < B2; ++b) {
                const int j = t + b * C::T;
#pragma unroll
                for (int r = 0; r < R2 / 2; ++r) {
                    const float2 x = sb[spad<C::LP>(j + (r + h * (R2 / 2)) * S2 - h * HN) * C::SS];
                    if (h == 0)
                        lo[b][r] = x;
                    else
                        v[b * R2 + R2 / 2 + r] = x;
                }
            }
        }
#pragma unroll
        for (int b = 0; b < B2; ++b) {
#pragma unroll
            for (int r = 0; r < R2 / 2; ++r) v[b * R2 + r] = lo[b][r];
        }
#pragma unroll
        for (int b = 0; b < B2; ++b) apply_twiddles<C, DIR, P + 1>(v + b * R2, pt[b]);
        run_passes_split<C, DIR, P + 1>(v, t, sb, tw);
    }
}

template <class RC, int DIR>
__global__ void __launch_bounds__(RC::C::THREADS, RC::MIN_CTAS)
    k_rows_big(const float2* in, float2* out, int64_t nrows, const float2* __restrict__ tw,
               int flags, int row_parity, int* err, uint64_t limit_ns) {
    using C = typename RC::C;
    constexpr int N = RC::N;
    extern __shared__ __align__(128) float2 smem[];
    float2* stage = smem;
    float2* xb = smem + N;
    __shared__ uint64_t bar;
    __shared__ int stage_bad;

    const int t = (int)threadIdx.x;
    const int64_t r0 = blockIdx.x, rstride = gridDim.x;

    auto issue = [&](int64_t row) {
        const bool ok = check_range(row * N, N, nrows * N, err);
        mbar_arrive_expect_tx(&bar, ok ? (uint32_t)RC::STAGE_BYTES : 0u);
        if (ok) bulk_load(stage, in + row * N, (uint32_t)RC::STAGE_BYTES, &bar);
    };

    if (t == 0) {
        stage_bad = stage_misaligned(smem, err);
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (stage_bad) return;  // uniform: never copy into a misaligned stage
    if (t == 0 && r0 < nrows) issue(r0);

    constexpr int R0 = C::radix(0);
    constexpr int B0 = C::E / R0;
    constexpr int S0 = C::N / R0;
    constexpr int RL = C::radix(C::NPASS - 1);
    constexpr int BL = C::E / RL;
    constexpr int SL = C::N / RL;

    for (int64_t it = 0;; ++it) {
        const int64_t row = r0 + it * rstride;
        if (row >= nrows) break;
        const bool ok = mbar_wait_bounded(&bar, (uint32_t)(it & 1), limit_ns);
        if (__syncthreads_or(!ok)) {
            if (t == 0) {
                if (err) atomicExch(err, KERR_WAIT_TIMEOUT);
                mbar_wait_bounded(&bar, (uint32_t)(it & 1), kDrainLimitNs);
            }
            return;
        }
        const int rp = row_parity ? (int)(row & 1) : 0;
        float2 v[C::E];
#pragma unroll
        for (int b = 0; b < B0; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < R0; ++r) {
                const int e = j + r * S0;
                float2 x = stage[e];
                if (flags & KF_CHESS_LOAD) x = neg_if(x, (e + rp) & 1);
                v[b * R0 + r] = x;
            }
        }
        __syncthreads();  // the stage has been read: refill it with the next row now
        if (t == 0) {
            const int64_t nr = row + rstride;
            if (nr < nrows) {
                fence_proxy_async_smem();
                issue(nr);
            }
        }

        run_passes_split<C, DIR, 0>(v, t, xb, tw);

        if (!check_range(row * N, N, nrows * N, err)) continue;
        float2* dst = out + row * N;
#pragma unroll
        for (int b = 0; b < BL; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < RL; ++r) {
                const int k = j + r * SL;
                float2 y = v[b * RL + r];
                if (flags & KF_CHESS_STORE) y = neg_if(y, (k + rp) & 1);
                y = scale_pow2(y, flags);
                stg_stream(dst + k, y);
            }
        }
    }
}

template <class RC, int DIR>
cudaError_t launch_rows_big(const float2* in, float2* out, int64_t nrows, const float2* tw,
                            int flags, int row_parity, int* err, uint64_t limit_ns,
                            cudaStream_t stream) {
    auto kern = k_rows_big<RC, DIR>;
    static LaunchCache cache;
    LaunchGeom geo;
    cudaError_t e = cache.get(
        [&](int dev, LaunchGeom* g) {
            return setup_persistent(kern, RC::C::THREADS, RC::SMEM_BYTES, dev, g);
        },
        &geo);
    if (e != cudaSuccess) return e;
    const int64_t resident = (int64_t)geo.per_sm * geo.num_sms;
    const int64_t grid = nrows < resident ? nrows : resident;
    if (grid <= 0) return cudaSuccess;
    kern<<<(unsigned)grid, RC::C::THREADS, RC::SMEM_BYTES, stream>>>(in, out, nrows, tw, flags,
                                                                     row_parity, err, limit_ns);
    return cudaGetLastError();
}

}  // namespace gbfft
