/*
 * gbfft.h - C ABI of the batched fp32 FFT library for one NVIDIA GB300 GPU (sm_103a).
 *
 * The library computes
 *
 *     X_k = sum_{j<n} x_j * exp(s * 2*pi*i * j*k / n),   s = -1 forward, s = +1 inverse,
 *
 * on batches of contiguous rows (dims = 1: power-of-two n, or any n up to 2^20) or images
 * (dims = 2, power-of-two sides, row-column: all rows, then all columns), unnormalised in both
 * directions unless a plan asks for 1/n (fft_plan_set_normalization).  This is the discrete Fourier
 * transform of Mota, "High Performance Fourier Transforms on GPUs with GLSL", §2.2 Eq. 5, with
 * the sign convention of its Eq. 5 / Algorithm 2 and the unnormalised inverse of the WGSL
 * Stockham kernels in "src/sht/wgsl/fourier.ts"; the 2-D form is Mota §2.7 Eq. 19.
 *
 * Data types: complex data are complex64, interleaved (re, im) float32 pairs, 8 bytes per
 * point; real rows are float32.  All pointers passed to exec calls are DEVICE pointers owned by
 * the caller, contiguous and 16-byte aligned.  The stream argument is a cudaStream_t passed as
 * void* (NULL = the legacy default stream).  Exec calls are asynchronous on that stream: they
 * validate their arguments on the host, enqueue kernels and return; they never synchronise.
 *
 * Errors: every function returns FFT_OK (0) or a negative status.  Argument errors are
 * detected on the host before anything is enqueued.  There is no CPU fallback: if the device
 * or the kernels are unavailable the call fails with FFT_ERR_CUDA.
 *
 * Thread-safety: distinct plans may be used concurrently.  One plan must not be executed on
 * two streams at the same time (its workspace is shared by its executions).
 */
#ifndef GBFFT_H
#define GBFFT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gbfft_plan_s* fft_plan; /* opaque; created and freed by the library */

/* Direction = sign s of the exponent (Mota §2.3.1 Algorithm 2 and its inverse remark). */
enum { FFT_FORWARD = -1, FFT_INVERSE = +1 };

/* Data layouts.
 * FFT_LAYOUT_C2C          complex rows [batch][n] (dims 1) or images [batch][n][n] (dims 2).
 * FFT_LAYOUT_REAL_ROWMAJOR real rows [batch][n] float32 <-> spectrum [batch][mmax+1] complex64.
 * FFT_LAYOUT_REAL_MMAJOR   real rows [batch][n] float32 <-> spectrum [mmax+1][batch] complex64,
 *                          i.e. coefficient m of row r at index m*batch + r, the fm[m*NLAT+ilat]
 *                          layout of fourier.ts (fftSynthWGSL / fftAnalysWGSL). */
enum { FFT_LAYOUT_C2C = 0, FFT_LAYOUT_REAL_ROWMAJOR = 1, FFT_LAYOUT_REAL_MMAJOR = 2 };

/* Status codes. */
enum {
    FFT_OK = 0,
    FFT_ERR_INVALID_ARG = -1,      /* NULL pointer, bad enum, batch < 1, wrong exec kind,
                                      shift with a real layout, band limit out of range */
    FFT_ERR_UNSUPPORTED_SIZE = -2, /* n outside the supported lengths (see fft_plan_create) */
    FFT_ERR_MISALIGNED = -3,       /* a data pointer is not 16-byte aligned */
    FFT_ERR_OOM = -4,              /* device allocation of tables or workspace failed */
    FFT_ERR_CUDA = -5,             /* a CUDA runtime call or kernel launch failed */
    FFT_ERR_TIMEOUT = -6,          /* a bounded device-side wait gave up (fft_plan_check) */
    FFT_ERR_BOUNDS = -7            /* checked build only (libgbfft_checked.so, compiled with
                                      -DGBFFT_CHECKED): a device-side index or copy-coordinate
                                      check failed and the access was skipped (fft_plan_check) */
};

/* Largest supported transform sizes. */
#define FFT_MAX_LOG2N_1D 24   /* n <= 2^24 for dims = 1, complex rows */
#define FFT_MAX_LOG2N_REAL 15 /* n <= 2^15 for the real layouts (one-pass n/2-point core) */
#define FFT_MAX_LOG2N_2D 12   /* n <= 2^12 per side for dims = 2 */
#define FFT_MAX_N_ANY_LENGTH 1048576 /* rows (dims 1, complex or real) whose length is not a power of two */

/*
 * fft_plan_create - plan a batched transform on the current CUDA device.
 *   n         transform length (dims 1) or image side (dims 2): a power of two with
 *             1 <= n <= 2^24 (dims 1, complex), 4 <= n <= 2^15 (real layouts),
 *             2 <= n <= 2^12 (dims 2); or, for rows (dims 1) only,
 *             any length 3 <= n <= FFT_MAX_N_ANY_LENGTH (complex rows and band-limited real
 *             rows, dims 1; for real rows this is the any-nphi role of the direct-sum 'dft'
 *             mode of fourier.ts).  Lengths n <= 8192 whose prime factors are 2, 3, 5 and 7
 *             run mixed-radix Stockham passes (radices 2, 3, 4, 5, 7, 8) in one kernel (the
 *             mixed-radix extension of the radix-2^k passes, Mota §2.3); rows of such
 *             lengths above 8192 run two mixed-radix passes, n = N1*N2 (columns with the
 *             four-step twiddle, then rows with a transposed store, through a plan workspace
 *             of batch*n complex64; real rows two per transform, the analysis with a third,
 *             unpack pass); every other length is computed as the chirp-z (Bluestein)
 *             transform X_k = c_k sum_j (x_j c_j) conj(c_{k-j}), c_j = exp(s*pi*i*j^2/n),
 *             through power-of-two FFTs of length m >= 2n - 1 (the same unnormalised DFT of
 *             Mota, "High Performance Fourier Transforms on GPUs with GLSL", 2.2 Eq. 5, for
 *             lengths the radix-2^k passes cannot split): in one kernel for n <= 8192, as
 *             six passes over a plan workspace of 2 * rows * m complex64 above that (chirp,
 *             four-step forward FFT, four-step inverse FFT with the filter on its first load,
 *             chirp).  Real rows above
 *             8192 points always take two rows per transform (fft_plan_set_real_pairing).
 *   batch     number of rows (dims 1) or images (dims 2), >= 1.
 *   dims      1 or 2 (2 only with FFT_LAYOUT_C2C).
 *   direction FFT_FORWARD or FFT_INVERSE.  Real layouts: FORWARD = analysis (R2C, exec with
 *             fft_exec_r2c), INVERSE = synthesis (C2R, exec with fft_exec_c2r).
 *   layout    FFT_LAYOUT_*.
 *   shift     0 or 1; C2C only; n even, or any length that is not a power of two.  Forward:
 *             the input is pre-multiplied by the chessboard (-1)^j (dims 1) or (-1)^(row+col)
 *             (dims 2), which for even n makes the output fftshift(X) ("The 1D fftshift in
 *             CUDA by chessboard multiplication", the chessboard section).  Inverse: the output
 *             is post-multiplied by the same chessboard, i.e. it is IFFT(ifftshift(X)), so
 *             inverse-shift(forward-shift(x)) = n*x (dims 1) or n^2*x (dims 2).  For odd n
 *             (mixed-radix and chirp-z paths) the factors are exp(+2*pi*i*j*h/n) on the
 *             forward load and exp(-2*pi*i*k*h/n) on the inverse store, h = (n-1)/2, with the
 *             same meaning (fftshift moves bin 0 to index h); they come from a plan table
 *             (folded into the chirp tables on the chirp-z path).
 *   out       receives the plan.
 * The plan allocates its device twiddle tables, its workspace (large 1-D sizes only) and a
 * device error word with cudaMalloc on the current device, and copies the tables (computed on
 * the host in double precision and rounded once to float) synchronously.
 * Test override: the environment variable GBFFT_FORCE_PATH, read at every plan creation and
 * query, set to "fourstep" plans C2C rows of 2^12 <= n <= 2^14 points (whose default is a
 * single kernel per row) as the two-pass four-step transform with N2 = 256, N1 = n/256, with a
 * workspace of batch*n complex64; "chirpz" plans the lengths whose default is the mixed-radix
 * kernel as chirp-z transforms; "default", "onepass" or unset leaves every choice at its
 * default; any other value makes plan creation and query return FFT_ERR_INVALID_ARG.
 * Returns FFT_OK, FFT_ERR_INVALID_ARG, FFT_ERR_UNSUPPORTED_SIZE, FFT_ERR_OOM or FFT_ERR_CUDA;
 * on error *out is set to NULL and nothing is left allocated.
 */
int fft_plan_create(int64_t n, int64_t batch, int dims, int direction, int layout, int shift,
                    fft_plan* out);

/*
 * fft_plan_create_2d - plan a batched 2-D C2C transform of rectangular images: batch images of
 * ny rows x nx columns, row-major, complex64 (Mota, "High Performance Fourier Transforms on
 * GPUs with GLSL", 2.7 Eq. 19: the nx-point transform of every row, then the ny-point
 * transform of every column).  nx and ny are powers of two with 2 <= nx, ny <= 2^12; shift
 * folds the 2-D fftshift in as the chessboard (-1)^(x+y) (forward load, inverse store).
 * Everything else (ownership, execution with fft_exec_c2c, errors) is as for fft_plan_create
 * with dims = 2, which is the square case ny = nx.
 */
int fft_plan_create_2d(int64_t nx, int64_t ny, int64_t batch, int direction, int shift,
                       fft_plan* out);

/* fft_plan_query_2d - host-only description of the plan fft_plan_create_2d would make (as
 * fft_plan_query); allocates nothing and touches no device. */
int fft_plan_query_2d(int64_t nx, int64_t ny, int64_t batch, int direction, int shift, char* buf,
                      size_t len);

/*
 * fft_plan_set_normalization - normalize = 1 scales the plan's output by 1/n (dims 1) or
 * 1/(nx*ny) (dims 2), the factor Mota, "High Performance Fourier Transforms on GPUs with
 * GLSL", puts on the inverse transform (2.2 Eq. 5; 2.7 for images), so that a normalised
 * inverse undoes the forward transform exactly; 0 (the default) leaves both directions
 * unnormalised.  The factor is applied in the last kernel's store (an exact power of two for
 * power-of-two sizes; folded into the store chirp for other lengths), at no extra pass.
 * C2C plans only.  Host call; for lengths that are not powers of two it rewrites a small plan
 * table with a synchronous copy, so call it before enqueueing work that uses the plan.
 * Returns FFT_OK, FFT_ERR_INVALID_ARG (NULL or real-layout plan, normalize not 0/1) or
 * FFT_ERR_CUDA.
 */
int fft_plan_set_normalization(fft_plan plan, int normalize);

/*
 * fft_plan_set_band_limit - set mmax for a real-layout plan: the analysis keeps m = 0..mmax,
 * the synthesis reads F_0..F_mmax and assembles the Hermitian spectrum X_0 = Re F_0,
 * X_m = F_m, X_{n-m} = conj F_m (fourier.ts header comment and fftSynthWGSL).  Requires
 * 0 <= 2*mmax <= n.  mmax = n/2 (even n) gives the full n/2 + 1 half spectrum with the Nyquist
 * bin, which is real and its own mirror: the analysis returns it with a zero imaginary part,
 * the synthesis uses Re F_{n/2} once.  The default is (n-1)/2 (n/2 - 1 for even n: the pages'
 * band limit, no Nyquist bin).  Host only.
 * Returns FFT_OK or FFT_ERR_INVALID_ARG (NULL plan, C2C plan, mmax out of range).
 */
int fft_plan_set_band_limit(fft_plan plan, int64_t mmax);

/*
 * fft_plan_set_real_pairing - for a real-layout plan, pairing = 1 transforms two real rows per
 * complex transform: rows 2p and 2p+1 are packed as y = x1 + i x2 and one n-point complex FFT
 * serves both (Mota, "High Performance Fourier Transforms on GPUs with GLSL", §2.6 Eq. 17-18:
 * X1_k = (Y_k + conj Y_{n-k})/2, X2_k = (Y_k - conj Y_{n-k})/(2i), and for the synthesis
 * Y_k = X1_k + i X2_k, x1 = Re y, x2 = Im y).  pairing = 0 (the default) takes one row per
 * n/2-point complex transform with the two-for-one recombination of "src/sht/wgsl/fourier.ts".
 * Both give the same spectra and rows (within fp32 rounding); the layouts, band limit and
 * argument rules of fft_exec_r2c / fft_exec_c2r are unchanged, and an odd batch pairs its last
 * row with a zero row that is never written.  Power-of-two plans take it for n <= 2^14 (one
 * CTA holds the n-point complex row); plans of other lengths (the chirp-z path) for every n.
 * Host only.  Returns FFT_OK, FFT_ERR_INVALID_ARG (NULL plan, C2C plan, pairing not 0/1) or
 * FFT_ERR_UNSUPPORTED_SIZE (power-of-two n > 2^14).
 */
int fft_plan_set_real_pairing(fft_plan plan, int pairing);

/*
 * fft_plan_set_wait_timeout - time limit, in nanoseconds, of every device-side wait of the
 * plan's kernels (waits for asynchronous bulk copies into shared memory).  A wait that runs out
 * makes its CTA record the failure in the plan's device error word, wait (for at most 1 s) for
 * its own copies still in flight, and exit; fft_plan_check then returns FFT_ERR_TIMEOUT and the
 * outputs of that execution are undefined.  The default is 2 s.  ns = 0 is a diagnostic setting
 * that makes every such wait give up at once without polling, which exercises this error path
 * without a real stall.  Host only.  Returns FFT_OK or FFT_ERR_INVALID_ARG (NULL plan).
 */
int fft_plan_set_wait_timeout(fft_plan plan, uint64_t ns);

/*
 * fft_plan_set_diagnostic - test hook.  mode = FFT_DIAG_INDEX_ONLY makes the plan's kernels
 * skip every butterfly, twiddle multiplication and real-row recombination, so that an execution
 * moves each input value, unchanged, through the load and store epilogues alone: the
 * chessboard sign flips, the four-step transposed store X[k1 + N1*k2], the Hermitian gather of
 * a synthesis, the pack and unpack of two real rows per transform, and the row-major or
 * m-major spectrum layouts.  A test compares those outputs bit for bit with the index maps of
 * an independent implementation; the results are not Fourier transforms.  Built in for the
 * one-pass 4096-point and four-step 2^15-point C2C plans, real plans of 4096 and 2^15 points,
 * and 4096-point real plans with two rows per transform.  mode = 0 restores normal
 * execution.  Host only.  Returns FFT_OK, FFT_ERR_INVALID_ARG (NULL plan, unknown mode) or
 * FFT_ERR_UNSUPPORTED_SIZE (another plan; its exec calls then also return that status while
 * the mode is set).
 */
#define FFT_DIAG_INDEX_ONLY 1
int fft_plan_set_diagnostic(fft_plan plan, int mode);

/* fft_plan_workspace_bytes - device bytes the plan holds besides its twiddle tables
 * (informational).  Returns FFT_OK or FFT_ERR_INVALID_ARG. */
int fft_plan_workspace_bytes(fft_plan plan, size_t* bytes);

/*
 * fft_plan_describe - write a one-line, NUL-terminated description of the plan's execution
 * path (kernels, radix sequence, launch geometry) into buf (at most len bytes).  Host only.
 * Returns FFT_OK or FFT_ERR_INVALID_ARG.
 */
int fft_plan_describe(fft_plan plan, char* buf, size_t len);

/*
 * fft_plan_query - host-only planning: describe the path fft_plan_create would choose for
 * these parameters, without touching any device.  Same validation and return codes as
 * fft_plan_create (minus the device errors).  buf may be NULL when len is 0.
 */
int fft_plan_query(int64_t n, int64_t batch, int dims, int direction, int layout, int shift,
                   char* buf, size_t len);

/*
 * fft_exec_c2c - run a C2C plan: out = transform(in).
 *   in, out  device pointers to batch*n (dims 1) or batch*n*n (dims 2) complex64 values;
 *            in == out (in place) is allowed; otherwise the ranges must not overlap.
 *   stream   cudaStream_t as void*.
 * Returns FFT_OK, FFT_ERR_INVALID_ARG (NULL, real-layout plan), FFT_ERR_MISALIGNED or
 * FFT_ERR_CUDA (launch failure).  Device faults surface at the caller's next synchronisation.
 */
int fft_exec_c2c(fft_plan plan, const void* in, void* out, void* stream);

/*
 * fft_exec_r2c - run a FORWARD real-layout plan (band-limited analysis, fftAnalysWGSL):
 * F_m = sum_j x_j exp(-2*pi*i*m*j/n), m = 0..mmax, for every row.
 *   in   device float32 [batch][n];  out  device complex64 spectrum in the plan's layout.
 *   in and out must not overlap.
 * Returns FFT_OK, FFT_ERR_INVALID_ARG, FFT_ERR_MISALIGNED or FFT_ERR_CUDA.
 */
int fft_exec_r2c(fft_plan plan, const float* in, void* out, void* stream);

/*
 * fft_exec_c2r - run an INVERSE real-layout plan (band-limited synthesis, fftSynthWGSL):
 * x_j = Re F_0 + 2 * sum_{m=1}^{mmax} Re(F_m exp(+2*pi*i*m*j/n)), for every row (Im F_0 is
 * ignored).
 *   in   device complex64 spectrum in the plan's layout;  out  device float32 [batch][n].
 *   in and out must not overlap.
 * Returns FFT_OK, FFT_ERR_INVALID_ARG, FFT_ERR_MISALIGNED or FFT_ERR_CUDA.
 */
int fft_exec_c2r(fft_plan plan, const void* in, float* out, void* stream);

/*
 * fft_plan_check - synchronise the device, then read and clear the plan's device error word.
 * Kernels that wait on device-side events give up after a bounded number of polls and set
 * this word instead of hanging.  Returns FFT_OK, FFT_ERR_TIMEOUT, FFT_ERR_INVALID_ARG,
 * FFT_ERR_BOUNDS (checked build only: an index check failed) or FFT_ERR_CUDA (the
 * synchronisation itself reported an error, or a copy stage was misaligned).
 */
int fft_plan_check(fft_plan plan);

/* fft_plan_destroy - free the plan and its device memory (synchronises the device first).
 * NULL is accepted and ignored.  Returns FFT_OK or FFT_ERR_CUDA. */
int fft_plan_destroy(fft_plan plan);

/*
 * fft_exec_c2c_noalloc - the batched 1-D C2C transform for callers that cannot allocate device
 * memory.  The pages have no counterpart of this call; it exists for integration.
 *
 * Some callers may not call cudaMalloc at all: code running inside a host application or
 * framework that owns every byte of device memory through its own allocator and forbids
 * direct allocation, and latency-bound processing loops that cannot afford cudaMalloc's
 * implicit device synchronisation and unbounded latency.  Plans allocate their tables and
 * workspace, so those callers cannot create one.  This entry point needs no plan: its scratch
 * buffer (the four-step intermediate) and its twiddle tables are fixed-size static device
 * arrays of the library (16 MiB + 512 KiB, held by every GPU that loads them until the
 * process exits), and the call allocates nothing.
 *
 *   n, batch   2^15 <= n <= 2^21 (power of two) and batch * n <= 2^21 (the scratch capacity);
 *              anything larger returns FFT_ERR_UNSUPPORTED_SIZE.
 *   direction, shift   as for fft_plan_create (C2C, dims 1).
 *   in, out, stream    as for fft_exec_c2c (device pointers, 16-byte aligned, in == out
 *              allowed); the output equals that of fft_exec_c2c on a plan of the same size.
 * Set-up: the first call on each device (with that device current) resolves the static
 * arrays' device addresses and uploads the twiddle tables with a synchronous copy; make that
 * first call before any stream capture.  Later calls only enqueue two kernels.
 * All calls share the one scratch array: calls that overlap on the GPU (on different streams
 * or threads) race and corrupt each other's results; serialise them.  The scratch keeps the
 * last call's contents, and nothing in it needs clearing (every element read is first
 * written by the same call).
 * Device-side waits are bounded (2 s).  A wait that gives up makes its kernel stop early (the
 * output is then undefined) and sets a static error word of the library on that device; the
 * word stays set until read.  The call itself returns before the kernels run, so it cannot
 * report this: call fft_exec_c2c_noalloc with n == 0 (every other argument but `stream` is
 * ignored) to synchronise `stream`, read and clear the word, and get FFT_ERR_TIMEOUT if any
 * earlier call on the current device timed out (FFT_OK otherwise).
 * Returns FFT_OK, FFT_ERR_INVALID_ARG, FFT_ERR_UNSUPPORTED_SIZE, FFT_ERR_MISALIGNED or
 * FFT_ERR_CUDA; the status form (n == 0) returns FFT_OK, FFT_ERR_TIMEOUT, FFT_ERR_BOUNDS
 * (checked build only) or FFT_ERR_CUDA.
 */
int fft_exec_c2c_noalloc(int64_t n, int64_t batch, int direction, int shift, const void* in,
                         void* out, void* stream);

/*
 * fft_shift - standalone fftshift / ifftshift by index rotation (the memory-move variants of
 * "The 1D fftshift in CUDA by chessboard multiplication", "What is fftshift?"): moves bin 0 to
 * the middle of every row or image, or (inverse) back.
 *   in, out   DEVICE pointers to batch complex64 arrays, 8-byte aligned (16-byte alignment
 *             enables 16-byte accesses); owned by the caller.  in == out (in place) is allowed
 *             when every rotated extent is even (nx for dims 1; nx and ny for dims 2): the
 *             rotation by half is then a swap and fftshift equals ifftshift.  Any other
 *             overlap is an error.
 *   nx, ny    row length; dims 1 requires ny == 1, dims 2 takes ny x nx row-major images
 *             (rectangular allowed).  Any extents >= 1, odd ones included.
 *   dims      1 (rows) or 2 (images: both axes rotate).
 *   inverse   0: fftshift, out[(y + ny/2) mod ny][(x + nx/2) mod nx] = in[y][x] (halves
 *             rounded down, numpy's convention); 1: ifftshift, the rotation back.
 *   stream    cudaStream_t; asynchronous, no host synchronisation.
 * The transform plans fold the same shift into their loads and stores (the chessboard for even
 * lengths); this call is for data that are already transformed.
 * Returns FFT_OK, FFT_ERR_INVALID_ARG, FFT_ERR_UNSUPPORTED_SIZE, FFT_ERR_MISALIGNED or
 * FFT_ERR_CUDA.
 */
int fft_shift(const void* in, void* out, int64_t nx, int64_t ny, int64_t batch, int dims,
              int inverse, void* stream);

/* fft_status_string - static description of a status code (never NULL). */
const char* fft_status_string(int status);

/* fft_version - library version as major*10000 + minor*100 + patch. */
int fft_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GBFFT_H */
