// Persistent one-pass row kernel with asynchronous bulk-copy prefetch.
//
// Same transform as k_fft over contiguous rows (Stockham radix-64 passes in registers, padded
// shared-memory exchanges), restructured so that HBM reads never wait for compute: the grid is
// a whole number of CTAs per SM, each CTA walks a strided sequence of row blocks (W rows of N
// points, W*N = 4096, 32 KiB; one row from 4096 points up), and one thread keeps NST blocks in
// flight with cp.async.bulk
// copies into NST shared-memory stages, each completing on its own mbarrier.  A stage that has
// been read into registers doubles as the exchange buffer of its block, and is refilled with
// the block NST iterations ahead once the block's results have been stored.  With one stage
// per CTA (the measured best at 4096 points) six CTAs share an SM and the copies of some
// overlap the compute of the others.
// Outputs go straight from registers to HBM (coalesced, streaming stores).
//
// Every mbarrier wait is bounded (limit_ns); on expiry the CTA records KERR_WAIT_TIMEOUT in the
// plan's error word, waits (again bounded) for its own copies still in flight, and exits.
#pragma once

#include "fft_kernel.cuh"
#include "tma.cuh"

namespace gbfft {

template <int LOG2N_, int MAXRB_, int NST_>
struct RowsTmaCfg {
    static constexpr int LOG2N = LOG2N_;
    static constexpr int LOG2W = LOG2N_ < 12 ? 12 - LOG2N_ : 0;  // W*N = 4096 points per block
    using C = FftCfg<LOG2N_, MAXRB_, LOG2W, true>;
    static constexpr int NST = NST_;
    static constexpr int N = C::N;
    static constexpr int W = C::W;
    static constexpr int SROW = C::SROW > C::N ? C::SROW : C::N;  // per-row stage slots
    static constexpr int STAGE = SROW * W;                          // float2 per stage
    static constexpr uint32_t BLOCK_BYTES = (uint32_t)W * N * 8u;
    static constexpr size_t SMEM_BYTES = (size_t)NST * STAGE * sizeof(float2);
    // CTAs per SM the register allocation must allow: at 4096 points the shared memory holds
    // six CTAs of 64 threads, and the registers must not allow fewer
    static constexpr int MIN_CTAS = LOG2N_ == 12 ? 6 : 1;
    static_assert((STAGE * sizeof(float2)) % 128 == 0, "stages stay 128-byte aligned");
};

// SCALE: the output scaling of normalised plans (flags' scale bits) is a separate
// instantiation, so that the unscaled kernel carries none of its code.  IDX: the index-only
// diagnostic (identity_passes in place of the radix passes), instantiated for 4096 points only.
template <class RC, int DIR, bool SCALE, bool IDX = false>
__global__ void __launch_bounds__(RC::C::THREADS, RC::MIN_CTAS)
    k_rows_tma(const float2* in, float2* out, int64_t nrows, const float2* __restrict__ tw,
               int flags, int row_parity, int* err, uint64_t limit_ns) {
    using C = typename RC::C;
    constexpr int NST = RC::NST;
    constexpr int N = RC::N;
    extern __shared__ __align__(128) float2 smem[];
    __shared__ uint64_t bars[NST];

    const int tid = (int)threadIdx.x;
    const int w = tid / C::T;
    const int t = tid % C::T;
    const int64_t nblocks = (nrows + RC::W - 1) / RC::W;
    const int64_t blk0 = blockIdx.x, bstride = gridDim.x;

    auto issue = [&](int s, int64_t blk) {  // never copy into a misaligned stage; the waits will give up
        const int64_t rows = nrows - blk * RC::W < RC::W ? nrows - blk * RC::W : RC::W;
        const uint32_t bytes = (uint32_t)rows * N * 8u;
        const bool ok = check_range(blk * RC::W * N, rows * N, nrows * N, err) &&
                        check_range(s * RC::STAGE, rows * N, NST * RC::STAGE, err);
        mbar_arrive_expect_tx(&bars[s], ok ? bytes : 0u);
        if (ok) bulk_load(smem + s * RC::STAGE, in + blk * RC::W * N, bytes, &bars[s]);
    };

    __shared__ int stage_bad;
    if (tid == 0) {
        stage_bad = stage_misaligned(smem, err);
        for (int s = 0; s < NST; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (stage_bad) return;  // uniform: never copy into a misaligned stage
    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            const int64_t blk = blk0 + s * bstride;
            if (blk < nblocks) issue(s, blk);
        }
    }

    constexpr int R0 = C::radix(0);
    constexpr int B0 = C::E / R0;
    constexpr int S0 = C::N / R0;
    constexpr int RL = C::radix(C::NPASS - 1);
    constexpr int BL = C::E / RL;
    constexpr int SL = C::N / RL;

    for (int64_t it = 0;; ++it) {
        const int64_t blk = blk0 + it * bstride;
        if (blk >= nblocks) break;
        const int s = (int)(it % NST);
        const uint32_t parity = (uint32_t)((it / NST) & 1);
        const bool ok = mbar_wait_bounded(&bars[s], parity, limit_ns);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                if (err) atomicExch(err, KERR_WAIT_TIMEOUT);
                for (int k = 0; k < NST; ++k) {  // copies still in flight: iterations it..it+NST-1
                    const int64_t ik = it + k;
                    if (blk0 + ik * bstride < nblocks)
                        mbar_wait_bounded(&bars[ik % NST], (uint32_t)((ik / NST) & 1),
                                          kDrainLimitNs);
                }
            }
            return;
        }

        float2* sbuf = smem + s * RC::STAGE;
        const int64_t row = blk * RC::W + w;
        const bool active = row < nrows;
        const int rp = row_parity ? (int)(row & 1) : 0;
        float2 v[C::E];
#pragma unroll
        for (int b = 0; b < B0; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < R0; ++r) {
                const int e = j + r * S0;
                float2 x = sbuf[w * N + e];  // dense block layout written by the bulk copy
                if (flags & KF_CHESS_LOAD) x = neg_if(x, (e + rp) & 1);
                v[b * R0 + r] = x;
            }
        }
        __syncthreads();  // the stage becomes this block's exchange buffer

        auto refill = [&]() {
            if (tid == 0) {
                const int64_t nb = blk0 + (it + NST) * bstride;
                if (nb < nblocks) {
                    fence_proxy_async_smem();
                    issue(s, nb);
                }
            }
        };
        if constexpr (IDX)
            identity_passes<C>(v, t, sbuf + w * RC::SROW);
        else
            run_passes<C, DIR, 0>(v, t, sbuf + w * RC::SROW, tw);

        if (active && check_range(row * N, N, nrows * N, err)) {
            float2* dst = out + row * N;
#pragma unroll
            for (int b = 0; b < BL; ++b) {
                const int j = t + b * C::T;
#pragma unroll
                for (int r = 0; r < RL; ++r) {
                    const int k = j + r * SL;
                    float2 y = v[b * RL + r];
                    if (flags & KF_CHESS_STORE) y = neg_if(y, (k + rp) & 1);
                    if constexpr (SCALE) y = scale_pow2(y, flags);
                    stg_stream(dst + k, y);
                }
            }
        }
        __syncthreads();  // every thread is done with the stage
        refill();
    }
}

template <class RC, int DIR>
cudaError_t launch_rows_tma(const float2* in, float2* out, int64_t nrows, const float2* tw,
                            int flags, int row_parity, int* err, uint64_t limit_ns,
                            cudaStream_t stream) {
    auto plain = k_rows_tma<RC, DIR, false>;
    auto scaled = k_rows_tma<RC, DIR, true>;
    auto kern = (flags >> KF_SCALE_SHIFT) ? scaled : plain;
    if (flags & KF_INDEX_ONLY) {
        if constexpr (RC::LOG2N == 12) {
            auto idx = k_rows_tma<RC, DIR, false, true>;
            static LaunchCache icache;
            LaunchGeom g;
            cudaError_t e = icache.get(
                [&](int dev, LaunchGeom* gg) {
                    return setup_persistent(idx, RC::C::THREADS, RC::SMEM_BYTES, dev, gg);
                },
                &g);
            if (e != cudaSuccess) return e;
            kern = idx;
        } else {
            return cudaErrorNotSupported;
        }
    }
    static LaunchCache cache;  // attributes and occupancy are per device
    LaunchGeom geo;
    cudaError_t e = cache.get(
        [&](int dev, LaunchGeom* g) {
            cudaError_t r = setup_persistent(scaled, RC::C::THREADS, RC::SMEM_BYTES, dev, g);
            return r == cudaSuccess ? setup_persistent(plain, RC::C::THREADS, RC::SMEM_BYTES, dev, g)
                                    : r;
        },
        &geo);
    if (e != cudaSuccess) return e;
    const int64_t nblocks = (nrows + RC::W - 1) / RC::W;
    const int64_t resident = (int64_t)geo.per_sm * geo.num_sms;
    const int64_t grid = nblocks < resident ? nblocks : resident;
    if (grid <= 0) return cudaSuccess;
    kern<<<(unsigned)grid, RC::C::THREADS, RC::SMEM_BYTES, stream>>>(in, out, nrows, tw, flags, row_parity,
                                                         err, limit_ns);
    return cudaGetLastError();
}

}  // namespace gbfft
