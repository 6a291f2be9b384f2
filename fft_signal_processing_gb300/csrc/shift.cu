// Standalone fftshift / ifftshift by index rotation (the memory-move variants that "The 1D
// fftshift in CUDA by chessboard multiplication" compares with the chessboard premultiply):
// rows of any length and ny x nx images, complex64, out of place for any extents and in place
// when every rotated extent is even.  Declared in include/gbfft.h (fft_shift).
//
// fftshift moves bin 0 to the middle: out[(y + sy) mod ny][(x + sx) mod nx] = in[y][x] with
// (sy, sx) = (ny/2, nx/2) rounded down; ifftshift is the rotation back.  Both kernels are pure
// data movement (16 bytes per point: one read, one write), so they are bound by HBM bandwidth.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gbfft.h"
#include "fft_common.cuh"
#include "launch_cache.cuh"

namespace gbfft {
namespace {

constexpr int kShiftThreads = 256;

// Out of place, one thread per output point (or pair of points) over the whole batch, so the
// work is spread evenly whatever the row length.  Output (b, y, x) reads input
// (b, (y - sy) mod ny, (x - sx) mod nx); with PAIRS two neighbouring points move as one 16-byte
// access (nx and sx even, both buffers 16-byte aligned); with POW2 (nx a power of two) the row
// and column come from a shift and a mask instead of a division.
template <bool PAIRS, bool POW2>
__global__ void __launch_bounds__(kShiftThreads)
    k_roll(const float2* __restrict__ in, float2* __restrict__ out, int64_t nx, int64_t ny,
           int64_t units, int64_t sx, int64_t sy, int log2nx) {
    constexpr int P = PAIRS ? 2 : 1;
    const int64_t stride = (int64_t)gridDim.x * kShiftThreads;
#pragma unroll 4
    for (int64_t u = (int64_t)blockIdx.x * kShiftThreads + threadIdx.x; u < units; u += stride) {
        const int64_t i = u * P;
        const int64_t row = POW2 ? i >> log2nx : i / nx;
        const int64_t x = POW2 ? i & (nx - 1) : i - row * nx;
        int64_t srow = row;
        if (ny > 1) {
            const int64_t b = row / ny, y = row - b * ny;
            srow = b * ny + (y >= sy ? y - sy : y - sy + ny);
        }
        const int64_t src = srow * nx + (x >= sx ? x - sx : x - sx + nx);
        if constexpr (PAIRS)
            stg_stream4(reinterpret_cast<float4*>(out + i),
                        ldg_stream4(reinterpret_cast<const float4*>(in + src)));
        else
            stg_stream(out + i, ldg_stream(in + src));
    }
}

// In place, every rotated extent even: the rotation by half an extent is an involution, so
// points are swapped in pairs.  Rows (ny == 1): x < nx/2 with x + nx/2.  Images: every point
// of the upper half (y < ny/2) with the diagonally opposite one (y + ny/2, (x + nx/2) mod nx).
// One warp per upper row; PAIRS as above (nx/2 even, buffer 16-byte aligned).
template <bool PAIRS>
__global__ void __launch_bounds__(kShiftThreads)
    k_swap_halves(float2* a, int64_t nx, int64_t ny, int64_t upper_rows) {
    const int lane = (int)threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * kShiftThreads + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * kShiftThreads) >> 5;
    const int64_t hx = nx / 2;
    const int64_t hy = ny / 2;
    const int64_t xend = ny == 1 ? hx : nx;  // rows: the first half; images: the whole row
    for (int64_t u = warp; u < upper_rows; u += nwarps) {
        int64_t r1, r2;
        if (ny == 1) {
            r1 = r2 = u;
        } else {
            const int64_t b = u / hy, y = u - b * hy;
            r1 = b * ny + y;
            r2 = r1 + hy;
        }
        float2* p1 = a + r1 * nx;
        float2* p2 = a + r2 * nx;
        if constexpr (PAIRS) {
#pragma unroll 2
            for (int64_t x = 2 * lane; x < xend; x += 64) {
                const int64_t x2 = x + hx < nx ? x + hx : x + hx - nx;
                float4* q1 = reinterpret_cast<float4*>(p1 + x);
                float4* q2 = reinterpret_cast<float4*>(p2 + x2);
                const float4 v1 = ldg_stream4(q1), v2 = ldg_stream4(q2);
                stg_stream4(q1, v2);
                stg_stream4(q2, v1);
            }
        } else {
#pragma unroll 2
            for (int64_t x = lane; x < xend; x += 32) {
                const int64_t x2 = x + hx < nx ? x + hx : x + hx - nx;
                const float2 v1 = ldg_stream(p1 + x), v2 = ldg_stream(p2 + x2);
                stg_stream(p1 + x, v2);
                stg_stream(p2 + x2, v1);
            }
        }
    }
}

unsigned grid_for(int64_t warps_needed) {
    static LaunchCache cache;  // the SM count of each device
    LaunchGeom geo;
    if (cache.get([](int dev, LaunchGeom* g) {
            return cudaDeviceGetAttribute(&g->num_sms, cudaDevAttrMultiProcessorCount, dev);
        },
                  &geo) != cudaSuccess)
        geo.num_sms = 1;
    const int num_sms = geo.num_sms;
    const int64_t blocks = (warps_needed * 32 + kShiftThreads - 1) / kShiftThreads;
    const int64_t cap = (int64_t)num_sms * 8;  // eight CTAs of 256 threads per SM
    return (unsigned)(blocks < cap ? (blocks < 1 ? 1 : blocks) : cap);
}

bool aligned(const void* p, uintptr_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

}  // namespace
}  // namespace gbfft

using namespace gbfft;

extern "C" int fft_shift(const void* in, void* out, int64_t nx, int64_t ny, int64_t batch,
                         int dims, int inverse, void* stream) {
    if (!in || !out || nx < 1 || ny < 1 || batch < 1) return FFT_ERR_INVALID_ARG;
    if ((dims != 1 && dims != 2) || (dims == 1 && ny != 1)) return FFT_ERR_INVALID_ARG;
    if (inverse != 0 && inverse != 1) return FFT_ERR_INVALID_ARG;
    if (nx > (INT64_C(1) << 40) / ny || batch > (INT64_C(1) << 58) / (nx * ny))
        return FFT_ERR_UNSUPPORTED_SIZE;
    if (!aligned(in, 8) || !aligned(out, 8)) return FFT_ERR_MISALIGNED;
    const int64_t points = batch * nx * ny;
    const uintptr_t a = (uintptr_t)in, b = (uintptr_t)out, bytes = (uintptr_t)points * 8u;
    const bool same = a == b;
    if (!same && a < b + bytes && b < a + bytes) return FFT_ERR_INVALID_ARG;  // partial overlap
    cudaStream_t st = (cudaStream_t)stream;
    cudaError_t e;
    if (same) {
        if ((nx & 1) || (dims == 2 && (ny & 1))) return FFT_ERR_INVALID_ARG;
        // fftshift and ifftshift coincide when every extent is even
        const int64_t upper = dims == 1 ? batch : batch * (ny / 2);
        const bool pairs = ((nx / 2) % 2 == 0) && aligned(out, 16);
        const unsigned grid = grid_for(upper);
        if (pairs)
            k_swap_halves<true><<<grid, kShiftThreads, 0, st>>>((float2*)out, nx, ny, upper);
        else
            k_swap_halves<false><<<grid, kShiftThreads, 0, st>>>((float2*)out, nx, ny, upper);
        e = cudaGetLastError();
    } else {
        int64_t sx = nx / 2, sy = dims == 2 ? ny / 2 : 0;
        if (inverse) {
            sx = (nx - sx) % nx;
            sy = (ny - sy) % ny;
        }
        const bool pairs = (nx % 2 == 0) && (sx % 2 == 0) && aligned(in, 16) && aligned(out, 16);
        const bool pow2 = (nx & (nx - 1)) == 0;
        int log2nx = 0;
        while ((INT64_C(1) << log2nx) < nx) ++log2nx;
        const int64_t units = pairs ? points / 2 : points;
        const unsigned grid = grid_for((units + 31) / 32);
        const float2* x = (const float2*)in;
        float2* y = (float2*)out;
        auto kern = pairs ? (pow2 ? k_roll<true, true> : k_roll<true, false>)
                          : (pow2 ? k_roll<false, true> : k_roll<false, false>);
        kern<<<grid, kShiftThreads, 0, st>>>(x, y, nx, ny, units, sx, sy, log2nx);
        e = cudaGetLastError();
    }
    return e == cudaSuccess ? FFT_OK : FFT_ERR_CUDA;
}
