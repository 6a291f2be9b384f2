// fft_exec_c2c_noalloc: the large-n (four-step) batched C2C transform for callers that must not
// allocate device memory.  Its intermediate buffer and its twiddle tables live in file-scope
// __device__ arrays of fixed size instead of cudaMalloc'ed plan memory, so the call itself
// allocates nothing.  See include/gbfft.h for the contract.
//
// The transform is the library's four-step path (the same two kernels as a plan of the same
// size): n = N1*N2 with N1 = 2^(l/2) and N2 = 2^(l - l/2); pass 1 writes N1-point column
// transforms times w_n^{n2*k1} into the scratch array, pass 2 reads it and writes the N2-point
// row transforms transposed into the output.  Pass 1 overwrites every scratch element that pass
// 2 reads, so the scratch never needs clearing between calls.
//
// Both kernels bound every device-side wait; a wait that gives up records KERR_WAIT_TIMEOUT in
// a file-scope error word (sticky until read), which the status form of the call (n == 0)
// reads and clears after synchronising the caller's stream.
#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "../../include/gbfft.h"
#include "fft_kernel.cuh"
#include "host_tables.h"
#include "kernels.h"
#include "tma.cuh"

using namespace gbfft;

static constexpr int kNoAllocMinLog2 = 15;  // below this the one-pass path needs no scratch
static constexpr int kNoAllocMaxLog2 = 21;
static constexpr int64_t kScratchPoints = int64_t(1) << 21;  // complex64 points: 16 MiB
static constexpr int kTableFloat2 = 1 << 16;                 // 512 KiB of twiddles, all sizes

// Every GPU that loads this module holds these until the process exits.
static __device__ __align__(256) float2 g_scratch[kScratchPoints];
static __device__ __align__(256) float2 g_tables[kTableFloat2];
static __device__ int g_err;  // KERR_* of a kernel that gave up, 0 otherwise

namespace {

constexpr int kMaxDevices = 64;
struct DeviceState {
    bool ready = false;
    float2* scratch = nullptr;  // device address of g_scratch on this device
    float2* tables = nullptr;   // device address of g_tables on this device
    int* err = nullptr;         // device address of g_err on this device
};
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

// Offsets (in float2) into g_tables of each size's sub-tables.
struct SizeTables {
    size_t col = 0, row = 0, hi = 0, lo = 0;
};
SizeTables g_off[kNoAllocMaxLog2 + 1];

// Host tables of every supported size, laid out once (identical on every device).
const std::vector<float2>& host_tables() {
    static std::vector<float2> v;
    static bool built = false;
    if (!built) {
        for (int l = kNoAllocMinLog2; l <= kNoAllocMaxLog2; ++l) {
            const int l1 = l / 2, l2 = l - l / 2, lowbits = (l + 1) / 2;
            g_off[l].col = host::append_pass_tables(v, l1, cols_pass_maxrb(l1, l - l1));
            g_off[l].row = host::append_pass_tables(v, l2, rowst_maxrb(l2));
            g_off[l].hi = host::append_roots(v, int64_t(1) << (l - lowbits),
                                             int64_t(1) << lowbits, int64_t(1) << l);
            g_off[l].lo = host::append_roots(v, int64_t(1) << lowbits, 1, int64_t(1) << l);
        }
        host::align_table(v);
        built = true;
    }
    return v;
}

// Once per device, with that device current: resolve the arrays' device addresses (host code
// must not use the array symbols themselves as pointers) and upload the twiddle tables.
int setup_device(int dev, DeviceState** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& st = g_dev[dev];
    if (!st.ready) {
        const std::vector<float2>& t = host_tables();
        if (t.size() > (size_t)kTableFloat2) return FFT_ERR_UNSUPPORTED_SIZE;
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess) return FFT_ERR_CUDA;
        st.scratch = (float2*)p;
        if (cudaGetSymbolAddress(&p, g_tables) != cudaSuccess) return FFT_ERR_CUDA;
        st.tables = (float2*)p;
        if (cudaGetSymbolAddress(&p, g_err) != cudaSuccess) return FFT_ERR_CUDA;
        st.err = (int*)p;
        if (cudaMemset(st.err, 0, sizeof(int)) != cudaSuccess) return FFT_ERR_CUDA;
        if (cudaMemcpy(st.tables, t.data(), t.size() * sizeof(float2), cudaMemcpyHostToDevice) !=
            cudaSuccess)
            return FFT_ERR_CUDA;
        st.ready = true;
    }
    *out = &st;
    return FFT_OK;
}

// Status form: wait for the stream, then read and clear this device's error word.
int query_status(cudaStream_t s) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FFT_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return FFT_ERR_CUDA;
    int* err = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_dev[dev].ready) return FFT_OK;  // nothing ran on this device
        err = g_dev[dev].err;
    }
    int h = 0;
    if (cudaMemcpy(&h, err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return FFT_ERR_CUDA;
    if (h == 0) return FFT_OK;
    if (cudaMemset(err, 0, sizeof(int)) != cudaSuccess) return FFT_ERR_CUDA;
    return kerr_status(h);
}

}  // namespace

extern "C" int fft_exec_c2c_noalloc(int64_t n, int64_t batch, int direction, int shift,
                                    const void* in, void* out, void* stream) {
    if (n == 0) return query_status((cudaStream_t)stream);
    if (!in || !out || batch < 1) return FFT_ERR_INVALID_ARG;
    if (direction != FFT_FORWARD && direction != FFT_INVERSE) return FFT_ERR_INVALID_ARG;
    if (shift != 0 && shift != 1) return FFT_ERR_INVALID_ARG;
    if (n < 1 || (n & (n - 1))) return FFT_ERR_UNSUPPORTED_SIZE;
    int l = 0;
    while ((int64_t(1) << l) < n) ++l;
    if (l < kNoAllocMinLog2 || l > kNoAllocMaxLog2) return FFT_ERR_UNSUPPORTED_SIZE;
    if (batch > kScratchPoints / n) return FFT_ERR_UNSUPPORTED_SIZE;  // scratch capacity
    if (((uintptr_t)in & 15u) || ((uintptr_t)out & 15u)) return FFT_ERR_MISALIGNED;
    const size_t bytes = (size_t)batch * (size_t)n * sizeof(float2);
    const uintptr_t a = (uintptr_t)in, b = (uintptr_t)out;
    if (in != out && a < b + bytes && b < a + bytes) return FFT_ERR_INVALID_ARG;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FFT_ERR_CUDA;
    DeviceState* st = nullptr;
    const int rc = setup_device(dev, &st);
    if (rc != FFT_OK) return rc;

    const int l1 = l / 2, l2 = l - l / 2, lowbits = (l + 1) / 2;
    const SizeTables& o = g_off[l];
    const bool fwd = direction == FFT_FORWARD;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = run_cols(l1, direction, (const float2*)in, st->scratch, batch << l2, l2,
                             st->tables + o.col, (shift && fwd) ? KF_CHESS_LOAD : 0, 0,
                             st->tables + o.hi, st->tables + o.lo, lowbits, st->err,
                             2000000000ull, s);
    if (e == cudaSuccess)
        e = run_rows_t(l2, direction, st->scratch, (float2*)out, batch << l1, l1,
                       st->tables + o.row, (shift && !fwd) ? KF_CHESS_STORE : 0, st->err,
                       2000000000ull, s);
    return e == cudaSuccess ? FFT_OK : FFT_ERR_CUDA;
}
