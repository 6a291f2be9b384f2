// Band-limited real rows: analysis (R2C) and synthesis (C2R) of N = 2^(LOG2H+1) real points
// through one H = N/2-point complex transform per row, with the two-for-one recombination
// fused into the kernel's load (synthesis) or store (analysis) phase.
//
// Semantics, from "src/sht/wgsl/fourier.ts" (header comment, fftSynthWGSL / fftAnalysWGSL):
//   analysis   F_m = sum_j x_j exp(-2*pi*i*m*j/N), m = 0..mmax, mmax < N/2;
//   synthesis  X_0 = Re F_0, X_m = F_m, X_{N-m} = conj F_m (1 <= m <= mmax), other bins 0,
//              x = inverse FFT of X (real), unnormalised.
// Recombination (the N/2-point real-FFT path of the same file):
//   analysis   z_m = x_{2m} + i x_{2m+1}, Z = FFT_H(z),
//              X_k = (Z_k + conj Z_{H-k})/2 - i e^{-2 pi i k/N} (Z_k - conj Z_{H-k})/2;
//   synthesis  Z_k = (X_k + conj X_{H-k}) + i e^{+2 pi i k/N} (X_k - conj X_{H-k}),
//              z = inverse FFT_H(Z), x_{2m} = Re z_m, x_{2m+1} = Im z_m,
// with Z_H = Z_0.  The Nyquist bin (mmax = H, even N only) is real and its own mirror:
// analysis X_H = Re Z_0 - Im Z_0; synthesis reads Re F_H into X_H (zero when mmax < H).
#pragma once

#include <cstring>

#include "cols_tma.cuh"
#include "fft_kernel.cuh"

namespace gbfft {

// The W rows of a CTA are adjacent lanes (thread = (w, t), w fastest) and interleaved in
// shared memory (slot i of row w at i*W + w), so spectrum gathers and scatters, the
// recombination and the radix exchanges all touch consecutive shared-memory words.
template <class C>
struct RealCfg {
    static_assert(!C::TFAST, "real kernels interleave their W rows");
    static constexpr int H = C::N;
    // per-row shared memory: the padded exchange, or H+1 slots for the recombination
    static constexpr int SLOTS = C::SROW > H + 1 ? C::SROW : H + 1;
    static constexpr size_t SMEM_BYTES = (size_t)SLOTS * C::W * sizeof(float2);
};

// R2C: in = real rows [nrows][2H] float32, out = spectrum (row-major [nrows][mmax+1] or
// m-major [mmax+1][nrows]).  twr[k] = (cos, sin)(2*pi*k/N), k < H.
// TMA = true (m-major spectrum, even row count): the spectrum tile [k][W] leaves through
// tensor stores of a 2-D map over (row, coefficient); coefficients above mmax are clipped by
// the map's extent.
// IDX: the index-only diagnostic: no core transform (identity_passes) and no recombination, so
// X_k = z_k (k < H) and X_H = z_0 land where the store epilogue puts them.
template <class C, bool TMA, bool IDX = false>
__global__ void __launch_bounds__(C::THREADS)
    k_r2c(const float* in, float2* out, int64_t nrows, int mmax, int mmajor,
          const float2* __restrict__ tw, const float2* __restrict__ twr,
          const __grid_constant__ CUtensorMap fmap, int* err) {
    constexpr int H = C::N;
    constexpr int W = C::W;
    extern __shared__ __align__(128) float2 smem[];
    const int w = (int)threadIdx.x % W;
    const int t = (int)threadIdx.x / W;
    const int64_t row0 = (int64_t)blockIdx.x * W;
    const int64_t row = row0 + w;
    const bool active = row < nrows;

    // z_m = x_{2m} + i x_{2m+1}: the real row read as H complex points
    constexpr int R0 = C::radix(0);
    constexpr int B0 = C::E / R0;
    constexpr int S0 = C::N / R0;
    float2 v[C::E];
    const bool inside = active && check_range(row * H, H, nrows * H, err);
    const float2* src = reinterpret_cast<const float2*>(in) + (inside ? row * H : 0);
#pragma unroll
    for (int b = 0; b < B0; ++b) {
        const int j = t + b * C::T;
#pragma unroll
        for (int r = 0; r < R0; ++r)
            v[b * R0 + r] = inside ? ldg_stream(src + j + r * S0) : make_float2(0.f, 0.f);
    }
    if constexpr (IDX)
        identity_passes<C>(v, t, smem + w);
    else
        run_passes<C, -1, 0>(v, t, smem + w, tw);

    constexpr int RL = C::radix(C::NPASS - 1);
    constexpr int BL = C::E / RL;
    constexpr int SL = C::N / RL;
    if constexpr (C::NPASS > 1) __syncthreads();  // last exchange fully read
#pragma unroll
    for (int b = 0; b < BL; ++b) {
        const int j = t + b * C::T;
#pragma unroll
        for (int r = 0; r < RL; ++r) smem[(j + r * SL) * W + w] = v[b * RL + r];  // Z_k
    }
    __syncthreads();

    // X_k = (Z_k + conj Z_{H-k})/2 - i e^{-i th_k} (Z_k - conj Z_{H-k})/2, k <= mmax
    auto recombine = [&](float2 zk, float2 zm, int k) {
        const float2 zc = make_float2(zm.x, -zm.y);                   // conj Z_{H-k}
        const float2 xe = make_float2(0.5f * (zk.x + zc.x), 0.5f * (zk.y + zc.y));
        const float2 d = make_float2(0.5f * (zk.x - zc.x), 0.5f * (zk.y - zc.y));
        const float2 xo = make_float2(d.y, -d.x);                     // -i * d
        return cadd(xe, ctw<-1>(xo, __ldg(twr + k)));                 // xe + e^{-i th} xo
    };
    if constexpr (TMA) {
        if (!tma_stage_aligned(smem, err)) return;
        // pairs {k, H-k}: one thread reads both Z's and writes both X's in place; threads
        // tid < W own k = 0 and keep Z_0 for the Nyquist bin
        constexpr int NB = H < 256 ? 1 : H / 256;
        constexpr int BK = H / NB;
        const float2 z0 = (int)threadIdx.x < W ? smem[threadIdx.x] : make_float2(0.f, 0.f);
        const int npair = IDX ? 0 : W * (H / 2 + 1);
        for (int i = (int)threadIdx.x; i < npair; i += C::THREADS) {
            const int wr = i % W, k = i / W;
            const int km = (H - k) & (H - 1);
            const float2 zk = smem[k * W + wr], zm = smem[km * W + wr];
            smem[k * W + wr] = recombine(zk, zm, k);
            if (km != k) smem[km * W + wr] = recombine(zm, zk, km);
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int b = 0; b < NB && b * BK <= mmax; ++b)
                if (check_box(row0, 1, nrows, b * BK, 1, mmax + 1, 0, 1, 8, err))
                    tma_store_2d(&fmap, (int)row0, b * BK, smem + b * BK * W);
            bulk_commit();
            bulk_wait_smem_read();  // shared memory stays valid until the stores have read it
        }
        if (mmax == H && (int)threadIdx.x < W && row0 + threadIdx.x < nrows &&  // X_H, real
            check_range((int64_t)H * nrows + row0 + threadIdx.x, 1, (int64_t)(mmax + 1) * nrows, err))
            stg_stream(out + (int64_t)H * nrows + row0 + threadIdx.x,
                       IDX ? z0 : make_float2(z0.x - z0.y, 0.f));
    } else {
        const int total = W * (mmax + 1);
#pragma unroll 4
        for (int i = (int)threadIdx.x; i < total; i += C::THREADS) {
            const int wr = i % W, k = i / W;
            const int64_t rr = row0 + wr;
            if (rr >= nrows) continue;
            float2 y;
            if (IDX) {
                y = smem[(k & (H - 1)) * W + wr];
            } else if (k == H) {  // Nyquist bin: Re Z_0 - Im Z_0
                const float2 z0 = smem[wr];
                y = make_float2(z0.x - z0.y, 0.f);
            } else {
                y = recombine(smem[k * W + wr], smem[((H - k) & (H - 1)) * W + wr], k);
            }
            const int64_t o = mmajor ? (int64_t)k * nrows + rr : rr * (mmax + 1) + k;
            if (check_range(o, 1, (int64_t)(mmax + 1) * nrows, err)) stg_stream(out + o, y);
        }
    }
}

// C2R: in = spectrum (layout as above), out = real rows [nrows][2H] float32.
// TMA = true (m-major spectrum, even row count): the spectrum tile [k][W] (k < H) arrives by
// tensor loads of a 2-D map over (row, coefficient); coefficients above mmax are filled with
// zeros by the copy engine.  The wait is bounded (limit_ns), reporting into *err.
// IDX: the index-only diagnostic: no recombination and no core transform, so
// x_{2k} = Re X_k, x_{2k+1} = Im X_k for the gathered X_k, k < H.
template <class C, bool TMA, bool IDX = false>
__global__ void __launch_bounds__(C::THREADS)
    k_c2r(const float2* in, float* out, int64_t nrows, int mmax, int mmajor,
          const float2* __restrict__ tw, const float2* __restrict__ twr,
          const __grid_constant__ CUtensorMap fmap, int* err, uint64_t limit_ns) {
    constexpr int H = C::N;
    constexpr int W = C::W;
    extern __shared__ __align__(128) float2 smem[];
    const int w = (int)threadIdx.x % W;
    const int t = (int)threadIdx.x / W;
    const int64_t row0 = (int64_t)blockIdx.x * W;
    const int64_t row = row0 + w;
    const bool active = row < nrows;

    // gather X_0..X_H (X_0 = Re F_0, zero above mmax, X_H = 0) as slots k*W + w
    if constexpr (TMA) {
        __shared__ uint64_t bar;
        constexpr int NB = H < 256 ? 1 : H / 256;
        constexpr int BK = H / NB;
        if (!tma_stage_aligned(smem, err)) return;
        if (threadIdx.x == 0) {
            prefetch_tensormap(&fmap);
            mbar_init(&bar, 1);
            fence_mbar_init();
            const bool ok = check_box(row0, 1, nrows, 0, NB * BK, H, 0, 1, 8, err);
            mbar_arrive_expect_tx(&bar, ok ? (uint32_t)(H * W * 8) : 0u);
            if (ok)
                for (int b = 0; b < NB; ++b) tma_load_2d(smem + b * BK * W, &fmap, (int)row0, b * BK, &bar);
        }
        __syncthreads();
        const bool ok = mbar_wait_bounded(&bar, 0, limit_ns);
        if (__syncthreads_or(!ok)) {
            if (threadIdx.x == 0) {
                if (err) atomicExch(err, KERR_WAIT_TIMEOUT);
                mbar_wait_bounded(&bar, 0, kDrainLimitNs);
            }
            return;
        }
        if (threadIdx.x < W) {
            smem[threadIdx.x].y = 0.f;  // X_0 = Re F_0
            // X_H = Re F_H with the Nyquist bin, else 0 (the tensor copies stop below H)
            float2 xh = make_float2(0.f, 0.f);
            if (mmax == H && row0 + threadIdx.x < nrows &&
                check_range((int64_t)H * nrows + row0 + threadIdx.x, 1, (int64_t)(mmax + 1) * nrows, err))
                xh.x = ldg_stream(in + (int64_t)H * nrows + row0 + threadIdx.x).x;
            smem[H * W + threadIdx.x] = xh;
        }
    } else {
        (void)err;
        (void)limit_ns;
        const int total = W * (H + 1);
#pragma unroll 8
        for (int i = (int)threadIdx.x; i < total; i += C::THREADS) {
            const int wr = i % W, k = i / W;
            const int64_t rr = row0 + wr;
            float2 x = make_float2(0.f, 0.f);
            const int64_t o = mmajor ? (int64_t)k * nrows + rr : rr * (mmax + 1) + k;
            if (rr < nrows && k <= mmax && check_range(o, 1, (int64_t)(mmax + 1) * nrows, err)) {
                x = ldg_stream(in + o);
                if (k == 0 || k == H) x.y = 0.f;  // X_0, X_H real
            }
            smem[k * W + wr] = x;
        }
    }
    __syncthreads();

    // Z_k = (X_k + conj X_{H-k}) + i e^{+i th_k} (X_k - conj X_{H-k}) for the first pass
    constexpr int R0 = C::radix(0);
    constexpr int B0 = C::E / R0;
    constexpr int S0 = C::N / R0;
    float2 v[C::E];
#pragma unroll
    for (int b = 0; b < B0; ++b) {
        const int j = t + b * C::T;
#pragma unroll
        for (int r = 0; r < R0; ++r) {
            const int k = j + r * S0;
            const float2 xk = smem[k * W + w];
            if (IDX) {
                v[b * R0 + r] = xk;
                continue;
            }
            const float2 xm = smem[(H - k) * W + w];
            const float2 xc = make_float2(xm.x, -xm.y);             // conj X_{H-k}
            const float2 sum = cadd(xk, xc);
            const float2 wd = ctw<+1>(csub(xk, xc), __ldg(twr + k));  // e^{+i th} (X_k - conj X_{H-k})
            v[b * R0 + r] = make_float2(sum.x - wd.y, sum.y + wd.x);  // sum + i * wd
        }
    }
    __syncthreads();  // the exchange buffer aliases the gathered spectrum

    if constexpr (IDX)
        identity_passes<C>(v, t, smem + w);
    else
        run_passes<C, +1, 0>(v, t, smem + w, tw);

    constexpr int RL = C::radix(C::NPASS - 1);
    constexpr int BL = C::E / RL;
    constexpr int SL = C::N / RL;
    if (active && check_range(row * H, H, nrows * H, err)) {
        float2* dst = reinterpret_cast<float2*>(out) + row * H;  // x_{2m}, x_{2m+1} = z_m
#pragma unroll
        for (int b = 0; b < BL; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < RL; ++r) stg_stream(dst + j + r * SL, v[b * RL + r]);
        }
    }
}

// Kernel attributes (dynamic shared memory above 48 KiB, maximum carveout) are set once per
// device and instantiation: Tag (the launch configuration) keeps one record per kernel.
template <class Tag, class K>
cudaError_t configure_once(K kern, size_t smem) {
    static LaunchCache cache;
    LaunchGeom geo;
    return cache.get(
        [&](int, LaunchGeom*) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            return e == cudaSuccess
                       ? cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100)
                       : e;
        },
        &geo);
}

// 2-D tensor map over an m-major spectrum [mmax+1][nrows]: (row, coefficient), box W x BK.
template <class C>
cudaError_t encode_spectrum_map(CUtensorMap* map, const void* base, int64_t nrows, int mmax) {
    constexpr int H = C::N;
    constexpr int NB = H < 256 ? 1 : H / 256;
    constexpr int BK = H / NB;
    EncodeTiledFn encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)nrows, (cuuint64_t)(mmax + 1)};
    const cuuint64_t strides[1] = {(cuuint64_t)nrows * 8u};
    const cuuint32_t box[2] = {(cuuint32_t)C::W, (cuuint32_t)BK};
    const cuuint32_t estr[2] = {1u, 1u};
    if (encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT64, 2, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    return cudaSuccess;
}

template <class C>
bool real_use_tma(int64_t nrows, int mmajor) {
    return mmajor && C::W >= 2 && (nrows % 2) == 0 && nrows >= C::W;
}

template <class C, bool IDX>
cudaError_t launch_r2c_impl(const float* in, float2* out, int64_t nrows, int mmax, int mmajor,
                            const float2* tw, const float2* twr, int* err, cudaStream_t stream) {
    constexpr size_t smem = RealCfg<C>::SMEM_BYTES;
    const int64_t grid = (nrows + C::W - 1) / C::W;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    CUtensorMap map;
    std::memset(&map, 0, sizeof map);
    if (real_use_tma<C>(nrows, mmajor)) {
        auto kern = k_r2c<C, true, IDX>;
        struct Tag {};
        cudaError_t e = configure_once<Tag>(kern, smem);
        if (e == cudaSuccess) e = encode_spectrum_map<C>(&map, out, nrows, mmax);
        if (e != cudaSuccess) return e;
        kern<<<(unsigned)grid, C::THREADS, smem, stream>>>(in, out, nrows, mmax, mmajor, tw, twr,
                                                            map, err);
    } else {
        auto kern = k_r2c<C, false, IDX>;
        struct Tag {};
        cudaError_t e = configure_once<Tag>(kern, smem);
        if (e != cudaSuccess) return e;
        kern<<<(unsigned)grid, C::THREADS, smem, stream>>>(in, out, nrows, mmax, mmajor, tw, twr,
                                                            map, err);
    }
    return cudaGetLastError();
}

template <class C, bool IDX>
cudaError_t launch_c2r_impl(const float2* in, float* out, int64_t nrows, int mmax, int mmajor,
                            const float2* tw, const float2* twr, int* err, uint64_t limit_ns,
                            cudaStream_t stream) {
    constexpr size_t smem = RealCfg<C>::SMEM_BYTES;
    const int64_t grid = (nrows + C::W - 1) / C::W;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    CUtensorMap map;
    std::memset(&map, 0, sizeof map);
    if (real_use_tma<C>(nrows, mmajor)) {
        auto kern = k_c2r<C, true, IDX>;
        struct Tag {};
        cudaError_t e = configure_once<Tag>(kern, smem);
        if (e == cudaSuccess) e = encode_spectrum_map<C>(&map, in, nrows, mmax);
        if (e != cudaSuccess) return e;
        kern<<<(unsigned)grid, C::THREADS, smem, stream>>>(in, out, nrows, mmax, mmajor, tw, twr,
                                                            map, err, limit_ns);
    } else {
        auto kern = k_c2r<C, false, IDX>;
        struct Tag {};
        cudaError_t e = configure_once<Tag>(kern, smem);
        if (e != cudaSuccess) return e;
        kern<<<(unsigned)grid, C::THREADS, smem, stream>>>(in, out, nrows, mmax, mmajor, tw, twr,
                                                            map, err, limit_ns);
    }
    return cudaGetLastError();
}

// ---- persistent kernels for the m-major spectrum (tensor copies) --------------------------------
// Real rows whose core is at most 2^11 points (the 2048 x 4096 real workload) are too few to
// fill the GPU in one wave of the kernels above, and each of those CTAs loads, transforms and
// stores in turn.  These persistent CTAs walk a strided sequence of tiles of W = 2 rows and keep
// the copy stage apart from the exchange area: as soon as a tile is in registers the next
// tile's copy is issued into the stage, so that it overlaps the transform and the stores.  C2R
// stages the spectrum tile [k][W] (k < H) by 2-D tensor copies (zero fill above mmax and past
// the last row); R2C stages W real rows by bulk copies into padded row slots and sends the
// spectrum out by tensor stores from the exchange area (clipped at mmax).  Every mbarrier wait
// is bounded; on expiry the CTA records KERR_WAIT_TIMEOUT, drains its copy and exits.
template <class C>
struct RealPCfg {
    static constexpr int H = C::N;
    static constexpr int W = C::W;
    static constexpr int SLOTS = C::SROW > H + 1 ? C::SROW : H + 1;
    static constexpr int WORK = SLOTS * W;                 // exchange area (float2)
    static constexpr int NB = H < 256 ? 1 : H / 256;       // tensor boxes per tile
    static constexpr int BK = H / NB;                      // coefficients per box
    static constexpr int C2R_STAGE = H * W;                // spectrum tile [k][W], k < H
    static constexpr int INROW = H + (W >= 8 ? 2 : 16 / W);  // padded real-row slot (float2)
    static constexpr int R2C_STAGE = W * INROW;
    static constexpr size_t C2R_SMEM = (size_t)(C2R_STAGE + WORK) * sizeof(float2);
    static constexpr size_t R2C_SMEM = (size_t)(R2C_STAGE + WORK) * sizeof(float2);
    static_assert(W >= 2, "tensor boxes are at least 16 bytes wide");
    static_assert((C2R_STAGE * 8) % 128 == 0 && (R2C_STAGE * 8) % 128 == 0,
                  "the exchange area stays 128-byte aligned");
};
// CTAs per SM the registers must allow: the shared memory holds three tiles' worth at the
// 2048-point core (67.6 KB each), and the synthesis would otherwise take 105 registers and run
// two CTAs per SM (80 registers at this bound, no spills).
constexpr int kRealPMinCtas = 3;

template <class C>
__global__ void __launch_bounds__(C::THREADS, kRealPMinCtas)
    k_c2r_p(const __grid_constant__ CUtensorMap fmap, const float2* in, float* out,
            int64_t nrows, int mmax, const float2* __restrict__ tw,
            const float2* __restrict__ twr, int* err, uint64_t limit_ns) {
    using P = RealPCfg<C>;
    constexpr int H = C::N;
    constexpr int W = C::W;
    extern __shared__ __align__(128) float2 smem[];
    float2* stage = smem;
    float2* work = smem + P::C2R_STAGE;
    __shared__ uint64_t bar;
    __shared__ int stage_bad;
    const int tid = (int)threadIdx.x;
    const int w = tid % W;
    const int t = tid / W;
    const int64_t ntiles = (nrows + W - 1) / W;
    const int64_t t0 = blockIdx.x, tstride = gridDim.x;

    auto issue = [&](int64_t tile) {  // the full box counts toward the bytes, OOB fill included
        const bool ok = check_box(tile * W, 1, nrows, 0, P::NB * P::BK, H, 0, 1, 8, err);
        mbar_arrive_expect_tx(&bar, ok ? (uint32_t)(H * W * 8) : 0u);
        if (!ok) return;
#pragma unroll 1
        for (int b = 0; b < P::NB; ++b)
            tma_load_2d(stage + b * P::BK * W, &fmap, (int)(tile * W), b * P::BK, &bar);
    };
    if (tid == 0) {
        stage_bad = stage_misaligned(stage, err) | stage_misaligned(work, err);
        prefetch_tensormap(&fmap);
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (stage_bad) return;  // uniform: never copy into a misaligned stage
    if (tid == 0 && t0 < ntiles) issue(t0);

    constexpr int R0 = C::radix(0);
    constexpr int B0 = C::E / R0;
    constexpr int S0 = C::N / R0;
    constexpr int RL = C::radix(C::NPASS - 1);
    constexpr int BL = C::E / RL;
    constexpr int SL = C::N / RL;
    for (int64_t it = 0;; ++it) {
        const int64_t tile = t0 + it * tstride;
        if (tile >= ntiles) break;
        const bool ok = mbar_wait_bounded(&bar, (uint32_t)(it & 1), limit_ns);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                if (err) atomicExch(err, KERR_WAIT_TIMEOUT);
                mbar_wait_bounded(&bar, (uint32_t)(it & 1), kDrainLimitNs);
            }
            return;
        }
        const int64_t row = tile * W + w;
        const bool active = row < nrows;
        // X_H: the Nyquist bin (real) when mmax = H, else 0 (the stage holds k < H)
        float2 xh = make_float2(0.f, 0.f);
        if (mmax == H && active &&
            check_range((int64_t)H * nrows + row, 1, (int64_t)(mmax + 1) * nrows, err))
            xh.x = ldg_stream(in + (int64_t)H * nrows + row).x;
        // Z_k = (X_k + conj X_{H-k}) + i e^{+i th_k} (X_k - conj X_{H-k}), X_0 real
        float2 v[C::E];
#pragma unroll
        for (int b = 0; b < B0; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < R0; ++r) {
                const int k = j + r * S0;
                float2 xk = stage[k * W + w];
                if (k == 0) xk.y = 0.f;
                const float2 xm = k == 0 ? xh : stage[(H - k) * W + w];
                const float2 xc = make_float2(xm.x, -xm.y);
                const float2 sum = cadd(xk, xc);
                const float2 wd = ctw<+1>(csub(xk, xc), __ldg(twr + k));
                v[b * R0 + r] = make_float2(sum.x - wd.y, sum.y + wd.x);
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
        run_passes<C, +1, 0>(v, t, work + w, tw);
        if (active && check_range(row * H, H, nrows * H, err)) {
            float2* dst = reinterpret_cast<float2*>(out) + row * H;  // x_{2m}, x_{2m+1} = z_m
#pragma unroll
            for (int b = 0; b < BL; ++b) {
                const int j = t + b * C::T;
#pragma unroll
                for (int r = 0; r < RL; ++r) stg_stream(dst + j + r * SL, v[b * RL + r]);
            }
        }
    }
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, kRealPMinCtas)
    k_r2c_p(const float* in, float2* out, const __grid_constant__ CUtensorMap fmap,
            int64_t nrows, int mmax, const float2* __restrict__ tw,
            const float2* __restrict__ twr, int* err, uint64_t limit_ns) {
    using P = RealPCfg<C>;
    constexpr int H = C::N;
    constexpr int W = C::W;
    extern __shared__ __align__(128) float2 smem[];
    float2* stage = smem;
    float2* work = smem + P::R2C_STAGE;
    __shared__ uint64_t bar;
    __shared__ int stage_bad;
    const int tid = (int)threadIdx.x;
    const int w = tid % W;
    const int t = tid / W;
    const int64_t ntiles = (nrows + W - 1) / W;
    const int64_t t0 = blockIdx.x, tstride = gridDim.x;
    const float2* zin = reinterpret_cast<const float2*>(in);  // z_m = x_{2m} + i x_{2m+1}

    auto issue = [&](int64_t tile) {
        const int64_t r0 = tile * W;
        const int rows = nrows - r0 < W ? (int)(nrows - r0) : W;
        const bool ok = check_range(r0 * H, (int64_t)rows * H, nrows * H, err);
        mbar_arrive_expect_tx(&bar, ok ? (uint32_t)rows * H * 8u : 0u);
        if (!ok) return;
#pragma unroll 1
        for (int r = 0; r < rows; ++r)
            bulk_load(stage + r * P::INROW, zin + (r0 + r) * H, (uint32_t)H * 8u, &bar);
    };
    if (tid == 0) {
        stage_bad = stage_misaligned(stage, err) | stage_misaligned(work, err);
        prefetch_tensormap(&fmap);
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (stage_bad) return;  // uniform: never copy into a misaligned stage
    if (tid == 0 && t0 < ntiles) issue(t0);

    constexpr int R0 = C::radix(0);
    constexpr int B0 = C::E / R0;
    constexpr int S0 = C::N / R0;
    constexpr int RL = C::radix(C::NPASS - 1);
    constexpr int BL = C::E / RL;
    constexpr int SL = C::N / RL;
    auto recombine = [&](float2 zk, float2 zm, int k) {  // X_k from Z_k and Z_{H-k}
        const float2 zc = make_float2(zm.x, -zm.y);
        const float2 xe = make_float2(0.5f * (zk.x + zc.x), 0.5f * (zk.y + zc.y));
        const float2 d = make_float2(0.5f * (zk.x - zc.x), 0.5f * (zk.y - zc.y));
        const float2 xo = make_float2(d.y, -d.x);
        return cadd(xe, ctw<-1>(xo, __ldg(twr + k)));
    };
    for (int64_t it = 0;; ++it) {
        const int64_t tile = t0 + it * tstride;
        if (tile >= ntiles) break;
        const bool ok = mbar_wait_bounded(&bar, (uint32_t)(it & 1), limit_ns);
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                if (err) atomicExch(err, KERR_WAIT_TIMEOUT);
                mbar_wait_bounded(&bar, (uint32_t)(it & 1), kDrainLimitNs);
            }
            return;
        }
        const int64_t row0 = tile * W;
        const bool active = row0 + w < nrows;
        float2 v[C::E];
#pragma unroll
        for (int b = 0; b < B0; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < R0; ++r)
                v[b * R0 + r] = active ? stage[w * P::INROW + j + r * S0] : make_float2(0.f, 0.f);
        }
        // the stage has been read (and the previous tile's spectrum stores have read the
        // exchange area: thread 0 waited for them before arriving here): refill the stage now
        __syncthreads();
        if (tid == 0) {
            const int64_t nt = tile + tstride;
            if (nt < ntiles) {
                fence_proxy_async_smem();
                issue(nt);
            }
        }
        run_passes<C, -1, 0>(v, t, work + w, tw);
        if constexpr (C::NPASS > 1) __syncthreads();  // last exchange fully read
#pragma unroll
        for (int b = 0; b < BL; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < RL; ++r) work[(j + r * SL) * W + w] = v[b * RL + r];  // Z_k
        }
        __syncthreads();
        // pairs {k, H-k} recombined in place; threads tid < W keep Z_0 for the Nyquist bin
        const float2 z0 = tid < W ? work[tid] : make_float2(0.f, 0.f);
        const int npair = W * (H / 2 + 1);
        for (int i = tid; i < npair; i += C::THREADS) {
            const int wr = i % W, k = i / W;
            const int km = (H - k) & (H - 1);
            const float2 zk = work[k * W + wr], zm = work[km * W + wr];
            work[k * W + wr] = recombine(zk, zm, k);
            if (km != k) work[km * W + wr] = recombine(zm, zk, km);
        }
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            for (int b = 0; b < P::NB && b * P::BK <= mmax; ++b)
                if (check_box(row0, 1, nrows, b * P::BK, 1, mmax + 1, 0, 1, 8, err))
                    tma_store_2d(&fmap, (int)row0, b * P::BK, work + b * P::BK * W);
            bulk_commit();
            bulk_wait_smem_read();  // the exchange area may be rewritten once the stores read it
        }
        if (mmax == H && tid < W && row0 + tid < nrows &&  // X_H = Re Z_0 - Im Z_0, real
            check_range((int64_t)H * nrows + row0 + tid, 1, (int64_t)(mmax + 1) * nrows, err))
            stg_stream(out + (int64_t)H * nrows + row0 + tid, make_float2(z0.x - z0.y, 0.f));
    }
}

// Persistent launch: one CTA per resident slot, at most one per tile.
template <class C, class K, class... Args>
cudaError_t launch_real_p(K kern, size_t smem, int64_t nrows, cudaStream_t stream,
                          Args... args) {
    static LaunchCache cache;
    LaunchGeom geo;
    cudaError_t e = cache.get(
        [&](int dev, LaunchGeom* g) { return setup_persistent(kern, C::THREADS, smem, dev, g); },
        &geo);
    if (e != cudaSuccess) return e;
    const int64_t ntiles = (nrows + C::W - 1) / C::W;
    const int64_t resident = (int64_t)geo.per_sm * geo.num_sms;
    const int64_t grid = ntiles < resident ? ntiles : resident;
    if (grid <= 0) return cudaSuccess;
    kern<<<(unsigned)grid, C::THREADS, smem, stream>>>(args...);
    return cudaGetLastError();
}

// The index-only diagnostic (KF_INDEX_ONLY in flags) is instantiated for real rows of 4096 and
// 2^15 points only.
template <class C>
cudaError_t launch_r2c(const float* in, float2* out, int64_t nrows, int mmax, int mmajor,
                       const float2* tw, const float2* twr, int flags, int* err,
                       uint64_t limit_ns, cudaStream_t stream) {
    if (flags & KF_INDEX_ONLY) {
        if constexpr (C::LOG2N == 11 || C::LOG2N == 14)
            return launch_r2c_impl<C, true>(in, out, nrows, mmax, mmajor, tw, twr, err, stream);
        else
            return cudaErrorNotSupported;
    }
    if constexpr (kRealPersistent && C::LOG2N >= 8 && C::LOG2N <= 11) {
        using PC = FftCfg<C::LOG2N, C::MAXRB, 1, false>;  // two rows per tile
        if (real_use_tma<PC>(nrows, mmajor)) {
            CUtensorMap map;
            cudaError_t e = encode_spectrum_map<PC>(&map, out, nrows, mmax);
            if (e != cudaSuccess) return e;
            return launch_real_p<PC>(k_r2c_p<PC>, RealPCfg<PC>::R2C_SMEM, nrows, stream, in, out,
                                     map, nrows, mmax, tw, twr, err, limit_ns);
        }
    }
    return launch_r2c_impl<C, false>(in, out, nrows, mmax, mmajor, tw, twr, err, stream);
}

template <class C>
cudaError_t launch_c2r(const float2* in, float* out, int64_t nrows, int mmax, int mmajor,
                       const float2* tw, const float2* twr, int flags, int* err,
                       uint64_t limit_ns, cudaStream_t stream) {
    if (flags & KF_INDEX_ONLY) {
        if constexpr (C::LOG2N == 11 || C::LOG2N == 14)
            return launch_c2r_impl<C, true>(in, out, nrows, mmax, mmajor, tw, twr, err,
                                            limit_ns, stream);
        else
            return cudaErrorNotSupported;
    }
    if constexpr (kRealPersistent && C::LOG2N >= 8 && C::LOG2N <= 11) {
        using PC = FftCfg<C::LOG2N, C::MAXRB, 1, false>;  // two rows per tile
        if (real_use_tma<PC>(nrows, mmajor)) {
            CUtensorMap map;
            cudaError_t e = encode_spectrum_map<PC>(&map, in, nrows, mmax);
            if (e != cudaSuccess) return e;
            return launch_real_p<PC>(k_c2r_p<PC>, RealPCfg<PC>::C2R_SMEM, nrows, stream, map, in,
                                     out, nrows, mmax, tw, twr, err, limit_ns);
        }
    }
    return launch_c2r_impl<C, false>(in, out, nrows, mmax, mmajor, tw, twr, err, limit_ns,
                                     stream);
}

}  // namespace gbfft
