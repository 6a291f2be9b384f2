// Persistent column-tile kernel with TMA tensor staging (2-D column pass; four-step pass 1).
//
// The data are matrices [L rows][S columns] of complex64 stored back to back (nmat of them);
// every column gets an L-point transform.  A tile is W adjacent columns of one matrix
// (W*8 bytes of every row; W*L = 4096 points, at least 2 columns).  Each CTA walks a strided sequence of tiles; one thread loads a
// tile with L/BH tensor copies (cp.async.bulk.tensor.3d, box W x BH x 1 of a 3-D tensor map
// over (column, row, matrix)) into a shared-memory stage that completes on an mbarrier.  The
// copy engine does the strided gathering, so the SM issues one instruction per box instead of
// one load per row segment.  The stage lands dense ([row][W]), is read into registers, then
// doubles as the padded exchange buffer of the tile's transforms (Stockham radix passes as in
// fft_kernel.cuh, the W columns interleaved).  Results, optionally multiplied by the four-step
// twiddle w_{L*S}^{c*k1}, go back into the stage in the dense tile layout and leave with tensor
// stores (the copy engine writes the W-wide row runs), after which the stage is refilled with
// the next tile.  Several CTAs share an SM, so the copies of some overlap the compute of
// others.  Every mbarrier wait is bounded; on expiry the CTA records KERR_WAIT_TIMEOUT, drains
// its copy and exits.
#pragma once

#include <cuda.h>

#include "fft_kernel.cuh"
#include "tma.cuh"

namespace gbfft {

// 3-D tiled tensor copy global -> shared, completing on `bar`.  Coordinates are in elements
// (x = column, y = row, z = matrix); x * 8 bytes is a multiple of 16 by construction (x is a
// multiple of W >= 2).
__device__ __forceinline__ void tma_load_3d(void* dst_smem, const CUtensorMap* map, int x, int y,
                                            int z, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// 3-D tiled tensor copy shared -> global (bulk async group of the issuing thread).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, int x, int y, int z,
                                             const void* src_smem) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(z), "r"(smem_addr(src_smem))
        : "memory");
}
// 2-D tiled tensor copies (global -> shared on an mbarrier; shared -> global in a bulk group).
__device__ __forceinline__ void tma_load_2d(void* dst_smem, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst_smem)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y,
                                             const void* src_smem) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(smem_addr(src_smem))
        : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

template <int LOG2L_, int MAXRB_, int LOG2W_>
struct ColsTmaCfg {
    using C = FftCfg<LOG2L_, MAXRB_, LOG2W_, false>;  // the W columns are adjacent lanes
    static constexpr int L = C::N;
    static constexpr int W = C::W;
    static constexpr int BH = L < 256 ? L : 256;  // rows per tensor box
    static constexpr int NBOX = L / BH;
    static constexpr int STAGE = (C::SROW > L ? C::SROW : L) * W;  // float2
    static constexpr uint32_t TILE_BYTES = (uint32_t)L * W * 8u;
    static constexpr size_t SMEM_BYTES = (size_t)STAGE * sizeof(float2);
    // CTAs per SM the register allocation must allow: as many as the shared memory allows
    static constexpr int MIN_CTAS =
        SMEM_BYTES > 113 * 1024 ? 1 : (C::THREADS <= 128 ? 3 : (C::THREADS <= 256 ? 2 : 1));
    static_assert(W >= 2, "tensor boxes are at least 16 bytes wide");
    static_assert((BH * W * 8) % 128 == 0, "boxes stay 128-byte aligned in shared memory");
};

struct ColsTwiddle {
    const float2* hi;  // w_{L*S}^q = hi[q >> lowbits] * lo[q & lowmask]
    const float2* lo;
    int lowbits;
    const float2* pre = nullptr;  // optional: input element q of each transform times pre[q]
};

// w_M^q for q reduced modulo M = 2^log2m, from the two-level table of the plan.
__device__ __forceinline__ float2 root2(const ColsTwiddle& t, uint32_t q, uint32_t mask) {
    q &= mask;
    return cmul(__ldg(t.hi + (q >> t.lowbits)), __ldg(t.lo + (q & ((1u << t.lowbits) - 1u))));
}

// IDX: the index-only diagnostic (identity_passes in place of the radix passes, no four-step
// twiddle).  PRE: element q = row*S + column of each [L][S] transform is multiplied by
// twd.pre[q] on the load (the chirp-z filter, fused into the inverse FFT's first pass).
template <class RC, int DIR, bool TW, bool IDX = false, bool PRE = false>
__global__ void __launch_bounds__(RC::C::THREADS, RC::MIN_CTAS)
    k_cols_tma(const __grid_constant__ CUtensorMap imap, const __grid_constant__ CUtensorMap omap,
               int64_t nmat, int log2s, const float2* __restrict__ tw, int flags, int elem_parity,
               ColsTwiddle twd, int* err, uint64_t limit_ns) {
    using C = typename RC::C;
    constexpr int W = RC::W;
    constexpr int RBL = C::rbits(C::NPASS - 1);
    constexpr int RL = 1 << RBL;
    constexpr int BL = C::E / RL;
    constexpr int SL = C::N / RL;
    constexpr int TA = tw_lo_count(RBL);  // four-step twiddle split r = a + TA*b
    constexpr int TB = RL / TA;
    extern __shared__ __align__(128) float2 smem[];
    __shared__ uint64_t bar;
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
            tma_load_3d(smem + b * RC::BH * W, &imap, x, b * RC::BH, z, &bar);
    };

    __shared__ int stage_bad;
    if (tid == 0) {
        stage_bad = stage_misaligned(smem, err);
        prefetch_tensormap(&imap);
        prefetch_tensormap(&omap);
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
            // fac[a][w] = w_M^{c*SL*a}, fac[TA + b][w] = w_M^{c*SL*TA*b} (M = L*S); the barrier
            // after the stage read publishes them (and orders them after the previous tile's use)
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
                float2 xv = smem[e * W + w];  // dense [row][W] tile written by the copy engine
                if constexpr (PRE) {
                    const int64_t q = ((int64_t)e << log2s) + c;
                    if (check_range(q, 1, S << C::LOG2N, err)) xv = cmul(xv, __ldg(twd.pre + q));
                }
                if (flags & KF_CHESS_LOAD) xv = neg_if(xv, (e * elem_parity + cp) & 1);
                v[b * R0 + r] = xv;
            }
        }
        __syncthreads();  // the stage becomes the exchange buffer

        if constexpr (IDX)
            identity_passes<C>(v, t, smem + w);
        else
            run_passes<C, DIR, 0>(v, t, smem + w, tw);

        // Output k = j + r*SL of column c.  Four-step: times w_M^{c*k} (M = L*S), formed as
        // w^{c*j} * w^{c*SL*a} * w^{c*SL*TA*b} for r = a + TA*b: one table lookup per butterfly,
        // the per-column factors from shared memory.
        if constexpr (TW && !IDX) {
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
        __syncthreads();  // every thread has read the last exchange
#pragma unroll
        for (int b = 0; b < BL; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < RL; ++r) {
                const int k = j + r * SL;
                float2 y = v[b * RL + r];
                if (flags & KF_CHESS_STORE) y = neg_if(y, (k * elem_parity + cp) & 1);
                y = scale_pow2(y, flags);
                smem[k * W + w] = y;  // dense [row][W] tile for the copy engine
            }
        }
        fence_proxy_async_smem();  // make this thread's tile writes visible to the copy engine
        __syncthreads();
        if (tid == 0) {
            if (check_box(x, W, S, 0, RC::NBOX * RC::BH, C::N, z, nmat, 8, err)) {
#pragma unroll 1
                for (int b = 0; b < RC::NBOX; ++b)
                    tma_store_3d(&omap, x, b * RC::BH, z, smem + b * RC::BH * W);
            }
            bulk_commit();
            bulk_wait_smem_read();  // the stage may be refilled once the stores have read it
            const int64_t nt = tile + tstride;
            if (nt < ntiles) issue(nt);
        }
    }
}

// Encode the 3-D tensor map (column, row, matrix) of `base` and launch.  The map is encoded
// per call on the host (it holds the global address).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn tensor_map_encoder();  // resolved once through the runtime (dispatch.cu)

template <class RC, int DIR, bool TW>
cudaError_t launch_cols_tma(const float2* in, float2* out, int64_t nmat, int log2s,
                            const float2* tw, int flags, int elem_parity, ColsTwiddle twd,
                            int* err, uint64_t limit_ns, cudaStream_t stream) {
    const auto plain = k_cols_tma<RC, DIR, TW>;
    auto kern = plain;
    if (twd.pre) {  // instantiated for the inverse column pass of the multi-pass chirp-z only
        if constexpr (TW && DIR > 0 && RC::L >= 128 && RC::L <= 1024) {
            kern = k_cols_tma<RC, DIR, TW, false, true>;
            static LaunchCache pcache;
            LaunchGeom g;
            cudaError_t e = pcache.get(
                [&](int dev, LaunchGeom* gg) {
                    return setup_persistent(kern, RC::C::THREADS, RC::SMEM_BYTES, dev, gg);
                },
                &g);
            if (e != cudaSuccess) return e;
        } else {
            return cudaErrorNotSupported;
        }
    }
    if (flags & KF_INDEX_ONLY) {  // instantiated for the 128-point pass of 2^15 only
        if constexpr (RC::L == 128) {
            kern = k_cols_tma<RC, DIR, TW, true>;
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
    EncodeTiledFn encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const int64_t S = int64_t(1) << log2s;
    if (S < RC::W) return cudaErrorInvalidValue;
    CUtensorMap imap, omap;
    const cuuint64_t dims[3] = {(cuuint64_t)S, (cuuint64_t)RC::L, (cuuint64_t)nmat};
    const cuuint64_t strides[2] = {(cuuint64_t)S * 8u, (cuuint64_t)S * RC::L * 8u};
    const cuuint32_t box[3] = {(cuuint32_t)RC::W, (cuuint32_t)RC::BH, 1u};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    for (int k = 0; k < 2; ++k) {
        if (encode(k == 0 ? &imap : &omap, CU_TENSOR_MAP_DATA_TYPE_FLOAT64, 3,
                   k == 0 ? const_cast<float2*>(in) : out, dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const int64_t ntiles = nmat * (S / RC::W);
    const int64_t resident = (int64_t)geo.per_sm * geo.num_sms;
    const int64_t grid = ntiles < resident ? ntiles : resident;
    if (grid <= 0) return cudaSuccess;
    kern<<<(unsigned)grid, RC::C::THREADS, RC::SMEM_BYTES, stream>>>(
        imap, omap, nmat, log2s, tw, flags, elem_parity, twd, err, limit_ns);
    return cudaGetLastError();
}

}  // namespace gbfft
