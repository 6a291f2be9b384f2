// The transform kernel: W independent power-of-two C2C transforms of N = 2^LOG2N points per
// CTA, each held in registers (E points per thread) and exchanged through padded shared
// memory between radix passes.  Where a transform's points live in HBM is described by a Map
// (contiguous rows, strided columns, or rows whose output is written transposed), so one
// kernel body serves the one-pass path, both passes of the four-step path and both passes of
// the 2-D path.
//
// Algorithm: Stockham autosort (natural order in and out, no bit reversal), decimation in
// time, as in the radix-2 / radix-4 Stockham kernels of "src/sht/wgsl/fourier.ts"
// (stockham(), stockham4()) and Mota, "High Performance Fourier Transforms on GPUs with
// GLSL", §2.5 (radix-4 Stockham), generalised to radix 64 per pass in registers (higher radix
// is the direction Mota §5.2 names as future work).  Pass p has radix R and span Ns (the
// product of the earlier radices).  Butterfly j (0 <= j < N/R) reads element j + r*N/R,
// r < R, multiplies element r by w_{Ns*R}^{(j mod Ns)*r}, does an R-point DFT in registers and
// writes element r to (j div Ns)*Ns*R + (j mod Ns) + r*Ns.  The first pass reads HBM directly
// and the last pass, where Ns = N/R, writes HBM at j + r*N/R; the passes in between exchange
// through shared memory.
#pragma once

#include "fft_common.cuh"

namespace gbfft {

// LOG2N: transform length; MAXRB: log2 of the largest radix per pass (registers per thread
// hold one butterfly of the first, largest radix); LOG2W: transforms per CTA; TFAST: lane order
// inside the CTA (true: a transform's threads are adjacent lanes, which suits contiguous rows;
// false: the W transforms are adjacent lanes, which suits columns and transposed stores
// because neighbouring transforms are neighbouring in memory).
template <int LOG2N_, int MAXRB_, int LOG2W_, bool TFAST_>
struct FftCfg {
    static constexpr int LOG2N = LOG2N_;
    static constexpr int MAXRB = MAXRB_;
    static constexpr int N = 1 << LOG2N;
    static constexpr int NPASS = sched_npass(LOG2N, MAXRB);
    static constexpr int LOG2E = sched_rbits(LOG2N, MAXRB, 0);
    static constexpr int E = 1 << LOG2E;  // points per thread = radix of the first pass
    static constexpr int T = N / E;       // threads per transform
    static constexpr int W = 1 << LOG2W_;
    static constexpr bool TFAST = TFAST_;
    static constexpr int THREADS = T * W;
    static constexpr int LP = LOG2E;  // shared-memory padding granularity (one slot per E)
    static constexpr int SROW = NPASS > 1 ? spad_size(N, LP) : 0;  // padded float2 per transform
    static constexpr size_t SMEM_BYTES = (size_t)SROW * W * sizeof(float2);
    // shared-memory element stride between consecutive (padded) indices of one transform
    static constexpr int SS = TFAST ? 1 : W;

    __host__ __device__ static constexpr int rbits(int p) { return sched_rbits(LOG2N, MAXRB, p); }
    __host__ __device__ static constexpr int radix(int p) { return 1 << rbits(p); }
    __host__ __device__ static constexpr int span(int p) {
        return 1 << sched_span_bits(LOG2N, MAXRB, p);
    }
};

// Twiddles of pass P for butterfly j: the A low and B high powers of w = w_{Ns*R}^(j mod Ns).
template <class C, int P>
struct PassTw {
    static constexpr int RB = C::rbits(P);
    static constexpr int A = tw_lo_count(RB);
    static constexpr int S = tw_stride(RB);
    float2 w[S];
};

template <class C, int P>
__device__ __forceinline__ void load_twiddles(PassTw<C, P>& pt, int j,
                                              const float2* __restrict__ tw) {
    constexpr int Ns = C::span(P);
    constexpr int S = PassTw<C, P>::S;
    const float4* w4 = reinterpret_cast<const float4*>(tw + tw_pass_off(C::LOG2N, C::MAXRB, P) +
                                                       (j & (Ns - 1)) * S);
#pragma unroll
    for (int i = 0; i < S / 2; ++i) {
        const float4 q = __ldg(w4 + i);
        pt.w[2 * i] = make_float2(q.x, q.y);
        pt.w[2 * i + 1] = make_float2(q.z, q.w);
    }
}

// v[r] *= w^r for r < R, with w^r = w^a * w^(A*b), r = a + A*b.
template <class C, int DIR, int P>
__device__ __forceinline__ void apply_twiddles(float2* v, const PassTw<C, P>& pt) {
    constexpr int R = C::radix(P);
    constexpr int A = PassTw<C, P>::A;
#pragma unroll
    for (int r = 1; r < R; ++r) {
        const int a = r % A, b = r / A;
        float2 f;
        if (b == 0)
            f = pt.w[a];
        else if (a == 0)
            f = pt.w[A + b];
        else
            f = cmul(pt.w[a], pt.w[A + b]);
        v[r] = ctw<DIR>(v[r], f);
    }
}

// Passes P..NPASS-1 on register data v (v[b*R + r] is element r of butterfly j = t + b*T);
// pass P's twiddles have already been applied.  sb points at this transform's first
// shared-memory slot; slots are C::SS apart.  The next pass's twiddles are fetched before the
// exchange barrier so that their latency hides behind it.
template <class C, int DIR, int P>
__device__ __forceinline__ void run_passes(float2 (&v)[C::E], int t, float2* sb,
                                           const float2* __restrict__ tw) {
    constexpr int R = C::radix(P);
    constexpr int B = C::E / R;
    constexpr int Ns = C::span(P);
#pragma unroll
    for (int b = 0; b < B; ++b) dft_reg<R, DIR>(v + b * R);
    if constexpr (P + 1 < C::NPASS) {
        if constexpr (P > 0) __syncthreads();  // every read of the previous exchange is done
#pragma unroll
        for (int b = 0; b < B; ++b) {
            const int j = t + b * C::T;
            const int base = (j / Ns) * Ns * R + (j & (Ns - 1));
#pragma unroll
            for (int r = 0; r < R; ++r) sb[spad<C::LP>(base + r * Ns) * C::SS] = v[b * R + r];
        }
        constexpr int R2 = C::radix(P + 1);
        constexpr int B2 = C::E / R2;
        constexpr int S2 = C::N / R2;
        PassTw<C, P + 1> pt[B2];
#pragma unroll
        for (int b = 0; b < B2; ++b) load_twiddles<C, P + 1>(pt[b], t + b * C::T, tw);
        __syncthreads();
#pragma unroll
        for (int b = 0; b < B2; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < R2; ++r) v[b * R2 + r] = sb[spad<C::LP>(j + r * S2) * C::SS];
            apply_twiddles<C, DIR, P + 1>(v + b * R2, pt[b]);
        }
        run_passes<C, DIR, P + 1>(v, t, sb, tw);
    }
}

// Index-only diagnostic (the bit-exact test of the load and store epilogues): in place of the
// radix passes, the values held in the first pass's register order (element j + r*N/R0 in
// v[b*R0 + r]) move unchanged into the last pass's order (element j + r*N/RL in v[b*RL + r])
// through the exchange buffer (sb: this transform's first slot, slots C::SS apart, room for the
// padded full length), so that the store epilogue writes element k where the load read it.
template <class C>
__device__ __forceinline__ void identity_passes(float2 (&v)[C::E], int t, float2* sb) {
    constexpr int R0 = C::radix(0);
    constexpr int RL = C::radix(C::NPASS - 1);
    if constexpr (R0 != RL) {
        constexpr int B0 = C::E / R0, S0 = C::N / R0;
        constexpr int BL = C::E / RL, SL = C::N / RL;
#pragma unroll
        for (int b = 0; b < B0; ++b) {
#pragma unroll
            for (int r = 0; r < R0; ++r)
                sb[spad<C::LP>(t + b * C::T + r * S0) * C::SS] = v[b * R0 + r];
        }
        __syncthreads();
#pragma unroll
        for (int b = 0; b < BL; ++b) {
#pragma unroll
            for (int r = 0; r < RL; ++r)
                v[b * RL + r] = sb[spad<C::LP>(t + b * C::T + r * SL) * C::SS];
        }
    }
}

// ---------------------------------------------------------------------------------------------
// Maps: where transform `tr` (0 <= tr < count) keeps its points.  Element e of the input is at
// in_base(tr) + e*in_stride(), element k of the output at out_base(tr) + k*out_stride().
// Chessboard parities: the sign of input element e is (-1)^(e*LE + lpar(tr)), of output
// element k is (-1)^(k*SE + spar(tr)).
// ---------------------------------------------------------------------------------------------

// Contiguous rows of N points (one-pass path; 2-D row pass with the row parity).
struct MapRows {
    int64_t count;
    int log2n;
    int row_parity;  // 1: include (-1)^row (2-D chessboard)
    __device__ int64_t in_base(int64_t tr) const { return tr << log2n; }
    __device__ int64_t out_base(int64_t tr) const { return tr << log2n; }
    __device__ int64_t in_stride() const { return 1; }
    __device__ int64_t out_stride() const { return 1; }
    static constexpr int LE = 1, SE = 1;
    __device__ int lpar(int64_t tr) const { return row_parity ? (int)(tr & 1) : 0; }
    __device__ int spar(int64_t tr) const { return row_parity ? (int)(tr & 1) : 0; }
    static constexpr bool TWIDDLE = false;
    __device__ float2 twiddle(int64_t, int) const { return make_float2(1.f, 0.f); }
};

// Columns of matrices [L][S] (S = 2^log2s columns, row stride S), stored back to back:
// transform tr is column c = tr mod S of matrix tr div S.  Used by the 2-D column pass (no
// twiddle; chessboard parity of column c) and by pass 1 of the four-step path (twiddle
// w_{L*S}^{c*k1} on output k1; the four-step chessboard parity is that of c, since
// n = n1*S + c with S even).
template <bool TW>
struct MapCols {
    int64_t count;
    int log2s, log2l;
    int elem_parity;                 // 1: element index enters the parity (2-D)
    const float2* __restrict__ hi;   // twiddle w_{L*S}^q = hi[q >> lowbits] * lo[q & lowmask]
    const float2* __restrict__ lo;
    int lowbits;
    __device__ int64_t in_base(int64_t tr) const {
        return ((tr >> log2s) << (log2s + log2l)) + (tr & ((1LL << log2s) - 1));
    }
    __device__ int64_t out_base(int64_t tr) const { return in_base(tr); }
    __device__ int64_t in_stride() const { return 1LL << log2s; }
    __device__ int64_t out_stride() const { return 1LL << log2s; }
    static constexpr int LE = 1, SE = 1;  // multiplied by elem_parity at use
    __device__ int lpar(int64_t tr) const { return (int)(tr & 1); }
    __device__ int spar(int64_t tr) const { return (int)(tr & 1); }
    static constexpr bool TWIDDLE = TW;
    __device__ float2 twiddle(int64_t tr, int k1) const {
        const uint32_t c = (uint32_t)(tr & ((1LL << log2s) - 1));
        const uint32_t q = (c * (uint32_t)k1) & ((1u << (log2s + log2l)) - 1u);
        return cmul(__ldg(hi + (q >> lowbits)), __ldg(lo + (q & ((1u << lowbits) - 1u))));
    }
};

// Rows of the four-step pass 2: transform tr = row k1 of matrix tr div N1 (N1 = 2^log2n1),
// input contiguous, output element k2 written to X[k1 + N1*k2] of its N1*N-point transform.
// Output parity (inverse chessboard) is that of k1, since k = k1 + N1*k2 with N1 even.
struct MapRowsT {
    int64_t count;
    int log2n, log2n1;
    __device__ int64_t in_base(int64_t tr) const { return tr << log2n; }
    __device__ int64_t out_base(int64_t tr) const {
        return ((tr >> log2n1) << (log2n1 + log2n)) + (tr & ((1LL << log2n1) - 1));
    }
    __device__ int64_t in_stride() const { return 1; }
    __device__ int64_t out_stride() const { return 1LL << log2n1; }
    static constexpr int LE = 0, SE = 0;
    __device__ int lpar(int64_t) const { return 0; }
    __device__ int spar(int64_t tr) const { return (int)(tr & 1); }
    static constexpr bool TWIDDLE = false;
    __device__ float2 twiddle(int64_t, int) const { return make_float2(1.f, 0.f); }
};

template <class M>
__device__ __forceinline__ int map_elem_parity(const M&) { return 1; }
template <>
__device__ __forceinline__ int map_elem_parity(const MapCols<false>& m) { return m.elem_parity; }
template <>
__device__ __forceinline__ int map_elem_parity(const MapCols<true>& m) { return m.elem_parity; }

// in == out is allowed for every map whose out_base/out_stride equal in_base/in_stride
// (rows, columns): each transform is read completely before any of it is written, and each
// transform belongs to exactly one CTA.
template <class C, int DIR, class M>
__global__ void __launch_bounds__(C::THREADS)
    k_fft(const float2* in, float2* out, M map, const float2* __restrict__ tw, int flags) {
    extern __shared__ float2 smem[];
    const int w = C::TFAST ? (int)threadIdx.x / C::T : (int)threadIdx.x % C::W;
    const int t = C::TFAST ? (int)threadIdx.x % C::T : (int)threadIdx.x / C::W;
    const int64_t tr = (int64_t)blockIdx.x * C::W + w;
    const bool active = tr < map.count;
    float2* sb = C::TFAST ? smem + w * C::SROW : smem + w;
    const int ep = map_elem_parity(map);

    constexpr int R0 = C::radix(0);
    constexpr int B0 = C::E / R0;
    constexpr int S0 = C::N / R0;
    float2 v[C::E];
    {
        const float2* src = in + (active ? map.in_base(tr) : 0);
        const int64_t is = map.in_stride();
        const int lp = map.lpar(tr);
#pragma unroll
        for (int b = 0; b < B0; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < R0; ++r) {
                const int e = j + r * S0;
                float2 x = active ? ldg_stream(src + e * is) : make_float2(0.f, 0.f);
                if (flags & KF_CHESS_LOAD) x = neg_if(x, (e * M::LE * ep + lp) & 1);
                v[b * R0 + r] = x;
            }
        }
    }

    run_passes<C, DIR, 0>(v, t, sb, tw);

    constexpr int RL = C::radix(C::NPASS - 1);
    constexpr int BL = C::E / RL;
    constexpr int SL = C::N / RL;
    if (active) {
        float2* dst = out + map.out_base(tr);
        const int64_t os = map.out_stride();
        const int sp = map.spar(tr);
#pragma unroll
        for (int b = 0; b < BL; ++b) {
            const int j = t + b * C::T;
#pragma unroll
            for (int r = 0; r < RL; ++r) {
                const int k = j + r * SL;
                float2 y = v[b * RL + r];
                if constexpr (M::TWIDDLE) y = ctw<DIR>(y, map.twiddle(tr, k));
                if (flags & KF_CHESS_STORE) y = neg_if(y, (k * M::SE * ep + sp) & 1);
                y = scale_pow2(y, flags);
                stg_stream(dst + k * os, y);
            }
        }
    }
}

template <class C, int DIR, class M>
cudaError_t launch_fft(const float2* in, float2* out, const M& map, const float2* tw, int flags,
                       cudaStream_t stream) {
    auto kern = k_fft<C, DIR, M>;
    if (C::SMEM_BYTES > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)C::SMEM_BYTES);
        if (e != cudaSuccess) return e;
    }
    const int64_t grid = (map.count + C::W - 1) / C::W;
    if (grid <= 0) return cudaSuccess;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, C::THREADS, C::SMEM_BYTES, stream>>>(in, out, map, tw, flags);
    return cudaGetLastError();
}

}  // namespace gbfft
