// Persistent four-step pass-2 kernel: row transforms with a transposed output, staged through
// shared memory by the copy engine in both directions.
//
// Pass 2 of the four-step transform (n = n1*N2 + n2, k = k1 + N1*k2) takes the N1 rows
// Y[k1][n2] of each transform, does the N2-point FFT of every row, and writes row k1's output
// k2 to X[k1 + N1*k2].  A block is W consecutive rows of one transform: W contiguous rows come
// in with W bulk copies into padded row slots of one shared-memory stage (padded so that
// reading the same element of the W rows hits distinct banks), the radix passes
// run with the W rows interleaved, and the results go back into the stage as a dense
// [k2][W] tile that leaves with tensor stores of a 3-D map over the output viewed as
// (k1, k2, transform): the copy engine writes the W-wide runs at stride N1.  One stage per CTA,
// several CTAs per SM; every mbarrier wait bounded.
#pragma once

#include "cols_tma.cuh"

namespace gbfft {

template <int LOG2N2_, int MAXRB_, int LOG2W_>
struct RowsTTmaCfg {
    using C = FftCfg<LOG2N2_, MAXRB_, LOG2W_, false>;  // the W rows are adjacent lanes
    static constexpr int N = C::N;
    static constexpr int W = C::W;
    // input row slot (float2, a 16-byte multiple): the W rows of one element index land in
    // distinct banks for the half-warp's 16/W values of t
    static constexpr int INROW = N + (W >= 8 ? 2 : 16 / W);
    static constexpr int BH = N < 256 ? N : 256;
    static constexpr int NBOX = N / BH;
    static constexpr int A1 = W * INROW;
    static constexpr int A2 = C::SROW * W;
    static constexpr int A3 = N * W;
    static constexpr int STAGE = ((A1 > A2 ? A1 : A2) > A3 ? (A1 > A2 ? A1 : A2) : A3);
    static constexpr uint32_t BLOCK_BYTES = (uint32_t)W * N * 8u;
    static constexpr size_t SMEM_BYTES = (size_t)STAGE * sizeof(float2);
    // CTAs per SM the register allocation must allow: as many as the shared memory allows
    static constexpr int MIN_CTAS =
        SMEM_BYTES > 113 * 1024 ? 1 : (C::THREADS <= 128 ? 3 : (C::THREADS <= 256 ? 2 : 1));
    static_assert(W >= 2, "tensor boxes are at least 16 bytes wide");
};

// IDX: the index-only diagnostic (identity_passes in place of the radix passes).
template <class RC, int DIR, bool IDX = false>
__global__ void __launch_bounds__(RC::C::THREADS, RC::MIN_CTAS)
    k_rowst_tma(const float2* in, const __grid_constant__ CUtensorMap omap, int64_t nrows,
                int log2n1, const float2* __restrict__ tw, int flags, int* err,
                uint64_t limit_ns) {
    using C = typename RC::C;
    constexpr int N = RC::N;
    constexpr int W = RC::W;
    extern __shared__ __align__(128) float2 smem[];
    __shared__ uint64_t bar;

    const int tid = (int)threadIdx.x;
    const int w = tid % W;
    const int t = tid / W;
    const int64_t nblocks = nrows / W;  // W divides N1, hence nrows
    const int64_t b0 = blockIdx.x, bstride = gridDim.x;
    const int64_t n1 = int64_t(1) << log2n1;

    auto issue = [&](int64_t blk) {
        const bool ok = check_range(blk * W * N, W * N, nrows * N, err);
        mbar_arrive_expect_tx(&bar, ok ? (uint32_t)RC::BLOCK_BYTES : 0u);
        if (!ok) return;
#pragma unroll 1
        for (int r = 0; r < W; ++r)
            bulk_load(smem + r * RC::INROW, in + (blk * W + r) * N, (uint32_t)N * 8u, &bar);
    };

    __shared__ int stage_bad;
    if (tid == 0) {
        stage_bad = stage_misaligned(smem, err);
        prefetch_tensormap(&omap);
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (stage_bad) return;  // uniform: never copy into a misaligned stage
    if (tid == 0 && b0 < nblocks) issue(b0);

    constexpr int R0 = C::radix(0);
    constexpr int B0 = C::E / R0;
    constexpr int S0 = C::N / R0;
    constexpr int RL = C::radix(C::NPASS - 1);
    constexpr int BL = C::E / RL;
    constexpr int SL = C::N / RL;

    for (int64_t it = 0;; ++it) {
        const int64_t blk = b0 + it * bstride;
        if (blk >= nblocks) break;
        const bool ok = mbar_wait_bounded(&bar, (uint32_t)(it & 1), limit_ns);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                if (err) atomicExch(err, KERR_WAIT_TIMEOUT);
                mbar_wait_bounded(&bar, (uint32_t)(it & 1), kDrainLimitNs);
            }
            return;
        }
        const int64_t row0 = blk * W;                     // first row k1 (global) of the block
        const int z = (int)(row0 >> log2n1);               // transform
        const int x = (int)(row0 & (n1 - 1));              // k1 of the block's first row
        const int rp = (int)((row0 + w) & 1);              // parity of k1 (N1 is even)

        float2 v[C::E];
#pragma unroll
        for (int b = 0; b < B0; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < R0; ++r) v[b * R0 + r] = smem[w * RC::INROW + j + r * S0];
        }
        __syncthreads();  // the stage becomes the exchange buffer

        if constexpr (IDX)
            identity_passes<C>(v, t, smem + w);
        else
            run_passes<C, DIR, 0>(v, t, smem + w, tw);

        __syncthreads();  // every thread has read the last exchange
#pragma unroll
        for (int b = 0; b < BL; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < RL; ++r) {
                const int k = j + r * SL;
                float2 y = v[b * RL + r];
                if (flags & KF_CHESS_STORE) y = neg_if(y, rp);
                y = scale_pow2(y, flags);
                smem[k * W + w] = y;  // dense [k2][W] tile for the copy engine
            }
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            if (check_box(x, W, n1, 0, RC::NBOX * RC::BH, N, z, nrows >> log2n1, 8, err)) {
#pragma unroll 1
                for (int b = 0; b < RC::NBOX; ++b)
                    tma_store_3d(&omap, x, b * RC::BH, z, smem + b * RC::BH * W);
            }
            bulk_commit();
            bulk_wait_smem_read();
            const int64_t nb = blk + bstride;
            if (nb < nblocks) issue(nb);
        }
    }
}

template <class RC, int DIR>
cudaError_t launch_rowst_tma(const float2* in, float2* out, int64_t nrows, int log2n1,
                             const float2* tw, int flags, int* err, uint64_t limit_ns,
                             cudaStream_t stream) {
    const auto plain = k_rowst_tma<RC, DIR>;
    auto kern = plain;
    if (flags & KF_INDEX_ONLY) {  // instantiated for the 256-point pass of 2^15 only
        if constexpr (RC::N == 256) {
            kern = k_rowst_tma<RC, DIR, true>;
            static LaunchCache icache;
            LaunchGeom g;
            cudaError_t e = icache.get(
                [&](int dev, LaunchGeom* gg) {
                    return setup_persistent(kern, RC::C::THREADS, RC::SMEM_BYTES, dev, gg);
                },
                &g);
            if (e != cudaSuccess) return e;
        } else {
            return cudaErrorNotSupported;
        }
    }
    static LaunchCache cache;
    LaunchGeom geo;
    cudaError_t e = cache.get(
        [&](int dev, LaunchGeom* g) {
            return setup_persistent(plain, RC::C::THREADS, RC::SMEM_BYTES, dev, g);
        },
        &geo);
    if (e != cudaSuccess) return e;
    const int64_t n1 = int64_t(1) << log2n1;
    if (n1 < RC::W || nrows % n1) return cudaErrorInvalidValue;
    EncodeTiledFn encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const int64_t nmat = nrows / n1;
    CUtensorMap omap;
    const cuuint64_t dims[3] = {(cuuint64_t)n1, (cuuint64_t)RC::N, (cuuint64_t)nmat};
    const cuuint64_t strides[2] = {(cuuint64_t)n1 * 8u, (cuuint64_t)n1 * RC::N * 8u};
    const cuuint32_t box[3] = {(cuuint32_t)RC::W, (cuuint32_t)RC::BH, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    if (encode(&omap, CU_TENSOR_MAP_DATA_TYPE_FLOAT64, 3, out, dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int64_t nblocks = nrows / RC::W;
    const int64_t resident = (int64_t)geo.per_sm * geo.num_sms;
    const int64_t grid = nblocks < resident ? nblocks : resident;
    if (grid <= 0) return cudaSuccess;
    kern<<<(unsigned)grid, RC::C::THREADS, RC::SMEM_BYTES, stream>>>(in, omap, nrows, log2n1, tw,
                                                                     flags, err, limit_ns);
    return cudaGetLastError();
}

}  // namespace gbfft
