// Persistent tile kernels for long strided transforms (column pass and transposed-row pass of
// 2048- and 4096-point transforms): the next tile's copy overlaps the whole transform of the
// current one.
//
// A tile of W = 4 transforms of 4096 points is 128 KB, so one CTA fills most of an SM's shared
// memory and a design in which the stage doubles as the exchange buffer (cols_tma.cuh,
// rowst_tma.cuh) leaves the SM idle while each tile is copied in and out.  Here the CTA keeps
// the stage and a half-length exchange buffer apart (the two-phase exchange of rows_big.cuh,
// with the W transforms interleaved lane by lane):
//   1. wait for the stage, read the tile into registers (first radix pass operands);
//   2. one thread issues the copy of the CTA's next tile into the stage at once;
//   3. radix passes through the exchange buffer;
//   4. results go straight from registers to HBM: lanes w = 0..W-1 of one output index write
//      one W*8-byte run (32 bytes at W = 4, a whole sector), so no staging is needed on the
//      way out and nothing waits for the stores.
// Column tiles arrive with 3-D tensor copies (column, row, matrix) like cols_tma.cuh; row
// blocks of the four-step pass 2 with one bulk copy per row into padded slots like
// rowst_tma.cuh.  Every mbarrier wait is bounded; on expiry the CTA records
// KERR_WAIT_TIMEOUT, drains its copy in flight and exits.
#pragma once

#include "cols_tma.cuh"
#include "rows_big.cuh"

namespace gbfft {

// ---- column pass --------------------------------------------------------------------------------
template <int LOG2L_, int MAXRB_, int LOG2W_>
struct ColsBigCfg {
    using C = FftCfg<LOG2L_, MAXRB_, LOG2W_, false>;  // the W columns are adjacent lanes
    static constexpr int L = C::N;
    static constexpr int W = C::W;
    static constexpr int BH = L < 256 ? L : 256;  // rows per tensor box
    static constexpr int NBOX = L / BH;
    static constexpr int STAGE = L * W;                          // dense [row][W] tile
    static constexpr int XCH = spad_size(L / 2, C::LP) * W;      // half-length exchange
    static constexpr uint32_t TILE_BYTES = (uint32_t)L * W * 8u;
    static constexpr size_t SMEM_BYTES = (size_t)(STAGE + XCH) * sizeof(float2);
    static constexpr int MIN_CTAS = SMEM_BYTES > 113 * 1024 ? 1 : 2;
    static_assert(C::NPASS >= 2, "long columns take several passes");
    static_assert(W >= 2, "tensor boxes are at least 16 bytes wide");
    static_assert((BH * W * 8) % 128 == 0, "boxes stay 128-byte aligned in shared memory");
};

template <class RC, int DIR, bool TW>
__global__ void __launch_bounds__(RC::C::THREADS, RC::MIN_CTAS)
    k_cols_big(const __grid_constant__ CUtensorMap imap, float2* out, int64_t nmat, int log2s,
               const float2* __restrict__ tw, int flags, int elem_parity, ColsTwiddle twd,
               int* err, uint64_t limit_ns) {
    using C = typename RC::C;
    constexpr int W = RC::W;
    constexpr int RBL = C::rbits(C::NPASS - 1);
    constexpr int RL = 1 << RBL;
    constexpr int BL = C::E / RL;
    constexpr int SL = C::N / RL;
    constexpr int TA = tw_lo_count(RBL);  // four-step twiddle split r = a + TA*b
    constexpr int TB = RL / TA;
    extern __shared__ __align__(128) float2 smem[];
    float2* stage = smem;
    float2* xb = smem + RC::STAGE;
    __shared__ uint64_t bar;
    __shared__ int stage_bad;
    __shared__ float2 fac[TW ? W * (TA + TB) : 1];  // four-step twiddle factors, [f][W]

    const int tid = (int)threadIdx.x;
    const int w = tid % W;
    const int t = tid / W;
    const int64_t S = int64_t(1) << log2s;
    const int64_t tiles_per_mat = S / W;
    const int64_t ntiles = nmat * tiles_per_mat;
    const int64_t t0 = blockIdx.x, tstride = gridDim.x;
    const uint32_t mask = (1u << (log2s + C::LOG2N)) - 1u;

    auto issue = [&](int64_t tile) {
        const int z = (int)(tile / tiles_per_mat);
        const int x = (int)((tile % tiles_per_mat) * W);
        const bool ok = check_box(x, W, S, 0, RC::NBOX * RC::BH, C::N, z, nmat, 8, err);
        mbar_arrive_expect_tx(&bar, ok ? (uint32_t)RC::TILE_BYTES : 0u);
        if (!ok) return;
#pragma unroll 1
        for (int b = 0; b < RC::NBOX; ++b)
            tma_load_3d(stage + b * RC::BH * W, &imap, x, b * RC::BH, z, &bar);
    };

    if (tid == 0) {
        stage_bad = stage_misaligned(stage, err);
        prefetch_tensormap(&imap);
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (stage_bad) return;  // uniform: never copy into a misaligned stage
    if (tid == 0 && t0 < ntiles) issue(t0);

    constexpr int R0 = C::radix(0);
    constexpr int B0 = C::E / R0;
    constexpr int S0 = C::N / R0;

    for (int64_t it = 0;; ++it) {
        const int64_t tile = t0 + it * tstride;
        if (tile >= ntiles) break;
        // (also the barrier after which the previous tile's factors may be overwritten)
        const bool ok = mbar_wait_bounded(&bar, (uint32_t)(it & 1), limit_ns);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                if (err) atomicExch(err, KERR_WAIT_TIMEOUT);
                mbar_wait_bounded(&bar, (uint32_t)(it & 1), kDrainLimitNs);  // the copy in flight
            }
            return;
        }
        const int z = (int)(tile / tiles_per_mat);
        const int x = (int)((tile % tiles_per_mat) * W);
        const uint32_t c = (uint32_t)x + (uint32_t)w;  // column of this thread's transform
        const int cp = (int)(c & 1);
        if constexpr (TW) {
            // fac[a][w] = w_M^{c*SL*a}, fac[TA + b][w] = w_M^{c*SL*TA*b} (M = L*S), published
            // by the barrier after the stage read
            for (int i = tid; i < W * (TA + TB); i += C::THREADS) {
                const uint32_t cw = (uint32_t)x + (uint32_t)(i % W);
                const int f = i / W;
                const uint32_t e = f < TA ? (uint32_t)(SL * f) : (uint32_t)(SL * TA * (f - TA));
                fac[i] = root2(twd, cw * e, mask);
            }
        }

        float2 v[C::E];
#pragma unroll
        for (int b = 0; b < B0; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < R0; ++r) {
                const int e = j + r * S0;
                float2 xv = stage[e * W + w];
                if (flags & KF_CHESS_LOAD) xv = neg_if(xv, (e * elem_parity + cp) & 1);
                v[b * R0 + r] = xv;
            }
        }
        __syncthreads();  // the stage has been read: refill it with the next tile now
        if (tid == 0) {
            const int64_t nt = tile + tstride;
            if (nt < ntiles) {
                fence_proxy_async_smem();
                issue(nt);
            }
        }

        run_passes_split<C, DIR, 0>(v, t, xb + w, tw);

        // Output k = j + r*SL of column c.  Four-step: times w_M^{c*k} (M = L*S), formed as
        // w^{c*j} * w^{c*SL*a} * w^{c*SL*TA*b} for r = a + TA*b.
        if constexpr (TW) {
            const float2* fw = fac + w;
#pragma unroll
            for (int b = 0; b < BL; ++b) {
                const uint32_t j = (uint32_t)(t + b * C::T);
                const float2 base = root2(twd, c * j, mask);
                float2 lb[TA];
                lb[0] = base;
#pragma unroll
                for (int a = 1; a < TA; ++a) lb[a] = cmul(base, fw[a * W]);
#pragma unroll
                for (int bb = 0; bb < TB; ++bb) {
                    const float2 hb = fw[(TA + bb) * W];
#pragma unroll
                    for (int a = 0; a < TA; ++a) {
                        const float2 f = bb == 0 ? lb[a] : cmul(lb[a], hb);
                        v[b * RL + a + TA * bb] = ctw<DIR>(v[b * RL + a + TA * bb], f);
                    }
                }
            }
        }
        if (!check_range(((int64_t)z << (log2s + C::LOG2N)) + c, 1, nmat << (log2s + C::LOG2N), err) ||
            !check_range(c, 1, S, err))
            continue;
        float2* dst = out + ((int64_t)z << (log2s + C::LOG2N)) + c;
#pragma unroll
        for (int b = 0; b < BL; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < RL; ++r) {
                const int k = j + r * SL;
                float2 y = v[b * RL + r];
                if (flags & KF_CHESS_STORE) y = neg_if(y, (k * elem_parity + cp) & 1);
                y = scale_pow2(y, flags);
                stg_stream(dst + ((int64_t)k << log2s), y);
            }
        }
    }
}

template <class RC, int DIR, bool TW>
cudaError_t launch_cols_big(const float2* in, float2* out, int64_t nmat, int log2s,
                            const float2* tw, int flags, int elem_parity, ColsTwiddle twd,
                            int* err, uint64_t limit_ns, cudaStream_t stream) {
    auto kern = k_cols_big<RC, DIR, TW>;
    static LaunchCache cache;
    LaunchGeom geo;
    cudaError_t e = cache.get(
        [&](int dev, LaunchGeom* g) {
            return setup_persistent(kern, RC::C::THREADS, RC::SMEM_BYTES, dev, g);
        },
        &geo);
    if (e != cudaSuccess) return e;
    EncodeTiledFn encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const int64_t S = int64_t(1) << log2s;
    if (S < RC::W) return cudaErrorInvalidValue;
    CUtensorMap imap;
    const cuuint64_t dims[3] = {(cuuint64_t)S, (cuuint64_t)RC::L, (cuuint64_t)nmat};
    const cuuint64_t strides[2] = {(cuuint64_t)S * 8u, (cuuint64_t)S * RC::L * 8u};
    const cuuint32_t box[3] = {(cuuint32_t)RC::W, (cuuint32_t)RC::BH, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    if (encode(&imap, CU_TENSOR_MAP_DATA_TYPE_FLOAT64, 3, const_cast<float2*>(in), dims,
               strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const int64_t ntiles = nmat * (S / RC::W);
    const int64_t resident = (int64_t)geo.per_sm * geo.num_sms;
    const int64_t grid = ntiles < resident ? ntiles : resident;
    if (grid <= 0) return cudaSuccess;
    kern<<<(unsigned)grid, RC::C::THREADS, RC::SMEM_BYTES, stream>>>(
        imap, out, nmat, log2s, tw, flags, elem_parity, twd, err, limit_ns);
    return cudaGetLastError();
}

// ---- four-step pass 2: rows in, transposed out ---------------------------------------------------
// Row k1 (of N1) of each transform gets an N-point FFT, its output k2 going to X[k1 + N1*k2].
// A block is W consecutive rows of one transform; lanes w of one output index write one run.
template <int LOG2N2_, int MAXRB_, int LOG2W_>
struct RowsTBigCfg {
    using C = FftCfg<LOG2N2_, MAXRB_, LOG2W_, false>;  // the W rows are adjacent lanes
    static constexpr int N = C::N;
    static constexpr int W = C::W;
    // input row slot (float2, a 16-byte multiple): element e of the W rows lands in distinct
    // banks for the half-warp's 16/W values of t
    static constexpr int INROW = N + (W >= 8 ? 2 : 16 / W);
    static constexpr int STAGE = W * INROW;
    static constexpr int XCH = spad_size(N / 2, C::LP) * W;  // half-length exchange
    static constexpr uint32_t BLOCK_BYTES = (uint32_t)W * N * 8u;
    static constexpr size_t SMEM_BYTES = (size_t)(STAGE + XCH) * sizeof(float2);
    static constexpr int MIN_CTAS = SMEM_BYTES > 113 * 1024 ? 1 : 2;
    static_assert(C::NPASS >= 2, "long rows take several passes");
    static_assert(W >= 2 && (INROW % 2) == 0, "row slots stay 16-byte aligned");
};

template <class RC, int DIR>
__global__ void __launch_bounds__(RC::C::THREADS, RC::MIN_CTAS)
    k_rowst_big(const float2* in, float2* out, int64_t nrows, int log2n1,
                const float2* __restrict__ tw, int flags, int* err, uint64_t limit_ns) {
    using C = typename RC::C;
    constexpr int N = RC::N;
    constexpr int W = RC::W;
    extern __shared__ __align__(128) float2 smem[];
    float2* stage = smem;
    float2* xb = smem + RC::STAGE;
    __shared__ uint64_t bar;
    __shared__ int stage_bad;

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
            bulk_load(stage + r * RC::INROW, in + (blk * W + r) * N, (uint32_t)N * 8u, &bar);
    };

    if (tid == 0) {
        stage_bad = stage_misaligned(stage, err);
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
        const int64_t row = blk * W + w;                  // this lane's row (global)
        const int64_t zt = row >> log2n1;                 // transform
        const int64_t k1 = row & (n1 - 1);
        const int rp = (int)(k1 & 1);                     // parity of k1 (N1 is even)

        float2 v[C::E];
#pragma unroll
        for (int b = 0; b < B0; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < R0; ++r) v[b * R0 + r] = stage[w * RC::INROW + j + r * S0];
        }
        __syncthreads();  // the stage has been read: refill it with the next block now
        if (tid == 0) {
            const int64_t nb = blk + bstride;
            if (nb < nblocks) {
                fence_proxy_async_smem();
                issue(nb);
            }
        }

        run_passes_split<C, DIR, 0>(v, t, xb + w, tw);

        // output k2 of this row lands at k1 + N1*k2 of its transform
        if (!check_range(((zt << log2n1) << C::LOG2N) + k1, (int64_t)(N - 1) * n1 + 1, nrows * N, err))
            continue;
        float2* dst = out + ((zt << log2n1) << C::LOG2N) + k1;
#pragma unroll
        for (int b = 0; b < BL; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < RL; ++r) {
                const int k = j + r * SL;
                float2 y = v[b * RL + r];
                if (flags & KF_CHESS_STORE) y = neg_if(y, rp);
                y = scale_pow2(y, flags);
                stg_stream(dst + ((int64_t)k << log2n1), y);
            }
        }
    }
}

template <class RC, int DIR>
cudaError_t launch_rowst_big(const float2* in, float2* out, int64_t nrows, int log2n1,
                             const float2* tw, int flags, int* err, uint64_t limit_ns,
                             cudaStream_t stream) {
    auto kern = k_rowst_big<RC, DIR>;
    static LaunchCache cache;
    LaunchGeom geo;
    cudaError_t e = cache.get(
        [&](int dev, LaunchGeom* g) {
            return setup_persistent(kern, RC::C::THREADS, RC::SMEM_BYTES, dev, g);
        },
        &geo);
    if (e != cudaSuccess) return e;
    const int64_t n1 = int64_t(1) << log2n1;
    if (n1 < RC::W || nrows % n1) return cudaErrorInvalidValue;
    const int64_t nblocks = nrows / RC::W;
    const int64_t resident = (int64_t)geo.per_sm * geo.num_sms;
    const int64_t grid = nblocks < resident ? nblocks : resident;
    if (grid <= 0) return cudaSuccess;
    kern<<<(unsigned)grid, RC::C::THREADS, RC::SMEM_BYTES, stream>>>(in, out, nrows, log2n1, tw,
                                                                     flags, err, limit_ns);
    return cudaGetLastError();
}

}  // namespace gbfft
