// C ABI of the library (declared in include/gbfft.h): plan creation and validation, the
// host-side planner, the fp64 twiddle tables, and the execution paths.
//
// Paths (chosen at plan creation, as the WGSL "src/sht/wgsl/fourier.ts" selects its 'fft' or
// 'dft' implementation at plan creation):
//   onepass   dims 1, n <= 2^14: one kernel, each row resident in one CTA.
//   fourstep  dims 1, 2^15 <= n <= 2^24 (from 2^12 when GBFFT_FORCE_PATH=fourstep):
//             n = N1*N2 with n = n1*N2 + n2 and k = k1 + N1*k2.
//             Pass 1 does the N1-point transforms down the N2 columns and multiplies output
//             (k1, n2) by w_n^{n2*k1}; pass 2 does the N2-point row transforms and writes row
//             k1's output k2 to X[k1 + N1*k2].  This is the four-step FFT the CS598 project page
//             ("Fast Fourier Transform on CPU and GPU") names for inputs that do not fit in
//             fast memory; the intermediate lives in the plan's workspace.
//   2d        n x n images: all rows, then all columns (Mota, "High Performance Fourier
//             Transforms on GPUs with GLSL", §2.7 Eq. 19), both in place in the output.
//   real      band-limited real rows through an n/2-point complex core (fourier.ts).
//   mixed     dims 1, complex or band-limited real rows of any length n <= 8192 that is not a
//             power of two but factors over {2, 3, 5, 7}: mixed-radix Stockham passes in one
//             kernel (mixed.cuh).
//   bluestein dims 1, complex or band-limited real rows of any other length n <= 8192 that is
//             not a power of two: the chirp-z transform through m-point FFTs (m >= 2n - 1) in
//             one kernel (bluestein.cuh); chirp and filter tables in double precision on the
//             host.  Longer rows: the same transform over four-step passes (bluestein_mp.cu).
//
// Twiddles are computed on the host in double precision from cos/sin of 2*pi*q/M with q
// reduced modulo M in integers, and rounded once to float (fourier.ts header comment: device
// trigonometry is too inaccurate for the fp32 transform error).
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "../../include/gbfft.h"
#include "fft_kernel.cuh"
#include "host_tables.h"
#include "kernels.h"
#include "mixed.h"
#include "tma.cuh"

using namespace gbfft;

namespace {

enum Path {
    PATH_ONEPASS = 0,
    PATH_FOURSTEP = 1,
    PATH_2D = 2,
    PATH_REAL = 3,
    PATH_BLUESTEIN = 4,
    PATH_BLUESTEIN_MP = 5,  // any length above kMaxBluesteinN: chirp-z over four-step passes
    PATH_MIXED = 6,         // lengths n <= kMaxMixedN with prime factors 2, 3, 5, 7 only
    PATH_MIXED_FS = 7,      // such lengths above kMaxMixedN (complex rows): two mixed-radix passes
};

struct PlanSpec {
    int64_t n = 0, batch = 0;
    int dims = 1, direction = -1, layout = 0, shift = 0;
    int log2n = 0;
    Path path = PATH_ONEPASS;
    int log2n1 = 0, log2n2 = 0;  // four-step split
    int nmix = 0;                // mixed-radix passes and their radices
    int mix_radix[kMaxMixedPasses] = {};
    int mix_n1 = 0, mix_n2 = 0;  // mixed-radix four-step split n = N1*N2
    int nmix1 = 0;               // ... and the N1-point schedule (the N2-point one in mix_radix)
    int mix_radix1[kMaxMixedPasses] = {};
    int lowbits = 0;             // four-step two-level twiddle split
    int log2m = 0;               // chirp-z transform length
    int64_t ny = 1;              // 2-D: rows per image (ny x n images; ny = n when square)
    int log2ny = 0;
};

// Test override of the path choice (environment variable GBFFT_FORCE_PATH, read at every plan
// creation or query): "fourstep" plans C2C rows of 2^12..2^14 points, whose default is the
// one-pass kernel, as the two-pass four-step transform (N2 = 2^8, N1 = n/2^8: the smallest
// split both passes serve); "chirpz" plans rows of lengths n <= kMaxMixedN whose default is the
// mixed-radix kernel as chirp-z transforms; "default" or unset keeps the default choice
// everywhere ("onepass" is accepted as a synonym).  Returns the FORCE_* value, or -1 for any
// other value.
enum { FORCE_NONE = 0, FORCE_FOURSTEP = 1, FORCE_CHIRPZ = 2 };
int forced_path() {
    const char* v = std::getenv("GBFFT_FORCE_PATH");
    if (!v || !*v || !std::strcmp(v, "default") || !std::strcmp(v, "onepass")) return FORCE_NONE;
    if (!std::strcmp(v, "fourstep")) return FORCE_FOURSTEP;
    if (!std::strcmp(v, "chirpz")) return FORCE_CHIRPZ;
    return -1;
}

// Radices of the mixed-radix schedule of n: the factors 7, 5 and 3 first (odd strides keep the
// first passes' shared-memory writes free of bank conflicts), then 8s and a last 4 or 2.
// Returns the number of passes, or 0 if n has a prime factor above 7.
int mixed_schedule(int64_t n, int* radix) {
    int np = 0;
    int64_t m = n;
    for (int r : {7, 5, 3})
        while (m % r == 0 && np < kMaxMixedPasses) {
            radix[np++] = r;
            m /= r;
        }
    while (m % 8 == 0 && np < kMaxMixedPasses) {
        radix[np++] = 8;
        m /= 8;
    }
    if ((m == 4 || m == 2) && np < kMaxMixedPasses) {
        radix[np++] = (int)m;
        m = 1;
    }
    return m == 1 ? np : 0;
}

// Four-step split of a length whose prime factors are 2, 3, 5, 7: the largest divisor N1 of n
// with N1 <= min(kMaxMixedN1, sqrt(n)) and N2 = n/N1 <= kMaxMixedN (both passes near the
// mixed-radix kernel's best lengths); 0 if there is none.
int mixed_split(int64_t n) {
    for (int64_t d = std::min<int64_t>(kMaxMixedN1, (int64_t)std::sqrt((double)n)); d >= 2; --d)
        if (n % d == 0 && n / d <= kMaxMixedN) return (int)d;
    return 0;
}
constexpr int kForcedFourStepMinLog2 = 12;  // N1 = 2^4 is the row pass's block of 16 rows
constexpr int kForcedFourStepLog2N2 = 8;    // the smallest four-step row pass

int ilog2_exact(int64_t n) {
    if (n < 1 || (n & (n - 1))) return -1;
    int l = 0;
    while ((int64_t(1) << l) < n) ++l;
    return l;
}

// Host validation and path choice shared by fft_plan_create and fft_plan_query.
// ny: rows per image for dims 2 (0 means square, ny = n); ignored for dims 1.
int plan_spec(int64_t n, int64_t batch, int dims, int direction, int layout, int shift,
              PlanSpec* ps, int64_t ny = 0) {
    if (batch < 1) return FFT_ERR_INVALID_ARG;
    if (dims != 1 && dims != 2) return FFT_ERR_INVALID_ARG;
    if (direction != FFT_FORWARD && direction != FFT_INVERSE) return FFT_ERR_INVALID_ARG;
    if (layout != FFT_LAYOUT_C2C && layout != FFT_LAYOUT_REAL_ROWMAJOR &&
        layout != FFT_LAYOUT_REAL_MMAJOR)
        return FFT_ERR_INVALID_ARG;
    if (shift != 0 && shift != 1) return FFT_ERR_INVALID_ARG;
    if (layout != FFT_LAYOUT_C2C && (dims != 1 || shift)) return FFT_ERR_INVALID_ARG;
    const int force = forced_path();
    if (force < 0) return FFT_ERR_INVALID_ARG;
    const int l = ilog2_exact(n);
    // lengths that are not powers of two: rows (complex or real) up to kMaxBluesteinMpN
    const bool any_length = l < 0 && dims == 1 && n >= 3 && n <= kMaxBluesteinMpN;
    if (l < 0 && !any_length) return FFT_ERR_UNSUPPORTED_SIZE;
    if (shift && (n & 1) && !any_length) return FFT_ERR_INVALID_ARG;
    PlanSpec s;
    s.n = n;
    s.batch = batch;
    s.dims = dims;
    s.direction = direction;
    s.layout = layout;
    s.shift = shift;
    s.log2n = l;
    int rad[kMaxMixedPasses], rad1[kMaxMixedPasses];
    const int nmix = any_length && n <= kMaxMixedN ? mixed_schedule(n, rad) : 0;
    // long rows: the split and both schedules (real rows two per transform)
    int n1 = 0, nmix1 = 0, nmix2 = 0;
    if (any_length && n > kMaxMixedN && n <= kMaxMixedFourStepN && force != FORCE_CHIRPZ &&
        (n1 = mixed_split(n)) > 0) {
        nmix1 = mixed_schedule(n1, rad1);
        nmix2 = mixed_schedule(n / n1, rad);
    }
    if (nmix > 0 && force != FORCE_CHIRPZ) {
        s.path = PATH_MIXED;
        s.nmix = nmix;
        for (int p = 0; p < nmix; ++p) s.mix_radix[p] = rad[p];
    } else if (nmix1 > 0 && nmix2 > 0) {
        s.path = PATH_MIXED_FS;
        s.mix_n1 = n1;
        s.mix_n2 = (int)(n / n1);
        s.nmix1 = nmix1;
        s.nmix = nmix2;
        for (int p = 0; p < nmix1; ++p) s.mix_radix1[p] = rad1[p];
        for (int p = 0; p < nmix2; ++p) s.mix_radix[p] = rad[p];
    } else if (any_length) {
        s.path = n <= kMaxBluesteinN ? PATH_BLUESTEIN : PATH_BLUESTEIN_MP;
        s.log2m = bluestein_log2m(n);
        s.log2n1 = s.log2m / 2;  // four-step split of the m-point transforms (multi-pass)
        s.log2n2 = s.log2m - s.log2m / 2;
        s.lowbits = (s.log2m + 1) / 2;
    } else if (layout != FFT_LAYOUT_C2C) {
        static_assert(FFT_MAX_LOG2N_REAL == kMaxLog2RealH + 1, "header and kernels agree");
        if (l < 2 || l > FFT_MAX_LOG2N_REAL) return FFT_ERR_UNSUPPORTED_SIZE;
        s.path = PATH_REAL;
    } else if (dims == 2) {
        if (l < 1 || l > FFT_MAX_LOG2N_2D) return FFT_ERR_UNSUPPORTED_SIZE;
        s.ny = ny ? ny : n;
        s.log2ny = ilog2_exact(s.ny);
        if (s.log2ny < 1 || s.log2ny > FFT_MAX_LOG2N_2D) return FFT_ERR_UNSUPPORTED_SIZE;
        s.path = PATH_2D;
    } else {
        if (l > FFT_MAX_LOG2N_1D) return FFT_ERR_UNSUPPORTED_SIZE;
        if (force == FORCE_FOURSTEP && l >= kForcedFourStepMinLog2 && l <= kMaxLog2OnePass) {
            s.path = PATH_FOURSTEP;
            s.log2n2 = kForcedFourStepLog2N2;
            s.log2n1 = l - kForcedFourStepLog2N2;
            s.lowbits = (l + 1) / 2;
        } else if (l <= kMaxLog2OnePass) {
            s.path = PATH_ONEPASS;
        } else {
            s.path = PATH_FOURSTEP;
            s.log2n1 = l / 2;      // column pass (strided)
            s.log2n2 = l - l / 2;  // row pass (contiguous in, transposed out)
            s.lowbits = (l + 1) / 2;
        }
    }
    // total element count must stay addressable with 64-bit byte offsets
    const int64_t per = dims == 2 ? n * s.ny : n;
    if (batch > (INT64_C(1) << 58) / per) return FFT_ERR_UNSUPPORTED_SIZE;
    *ps = s;
    return FFT_OK;
}

using host::append_pass_tables;
using host::append_roots;
using host::align_table;

std::string radix_string(int l, int maxrb) {
    std::string s;
    for (int p = 0; p < sched_npass(l, maxrb); ++p) {
        if (p) s += "x";
        s += std::to_string(1 << sched_rbits(l, maxrb, p));
    }
    return s;
}

struct Geo {
    int threads, per_cta;
    size_t smem;
};
size_t padded_bytes(int l, int maxrb, int w) {
    const int lp = sched_rbits(l, maxrb, 0);
    return sched_npass(l, maxrb) > 1 ? (size_t)spad_size(1 << l, lp) * (1u << w) * 8u : 0;
}
Geo rows_geo(int l) {
    if (l <= 4) return {256, 256, (size_t)256 * ((1 << l) + 1) * 8u};  // small-row kernel
    if (l >= kRowsTmaMinLog2 && l <= kRowsTmaMaxLog2) {  // persistent bulk-copy kernel
        const int w = 12 - l, lp = sched_rbits(l, rows_maxrb(l), 0);
        const size_t stage = (size_t)std::max(spad_size(1 << l, lp), 1 << l) * (1u << w) * 8u;
        return {(1 << rows_log2t(l)) << w, 1 << w, stage * kRowsTmaStages};
    }
    // long rows: full-row stage + half-row exchange buffer
    const int lp = sched_rbits(l, rows_maxrb(l), 0);
    return {1 << rows_log2t(l), 1,
            ((size_t)(1 << l) + (size_t)spad_size(1 << (l - 1), lp)) * 8u};
}
Geo cols_geo(int l, int log2s) {
    if (cols_use_big(l, log2s)) {  // tile stage + half-length exchange buffer
        const int w = cols_tma_log2w(l), lp = sched_rbits(l, cols_tma_maxrb(l), 0);
        const size_t b = ((size_t)(1 << l) + (size_t)spad_size(1 << (l - 1), lp)) << w;
        return {(1 << (l - lp)) << w, 1 << w, b * 8u};
    }
    if (cols_use_tma(l, log2s)) {
        const int w = cols_tma_log2w(l), lp = sched_rbits(l, cols_tma_maxrb(l), 0);
        const size_t stage = (size_t)std::max(spad_size(1 << l, lp), 1 << l) * (1u << w) * 8u;
        return {(1 << (l - lp)) << w, 1 << w, stage};
    }
    const int w = cols_log2w(l, 0);
    return {(1 << cols_log2t(l)) << w, 1 << w, padded_bytes(l, cols_maxrb(l), w)};
}
Geo rowst_geo(int l) {
    const int w = rowst_log2w(l), lp = sched_rbits(l, rowst_maxrb(l), 0);
    const size_t a = (size_t)((1 << l) + (w >= 3 ? 2 : 16 >> w)) << w;
    if (rowst_use_big(l))  // row slots + half-length exchange buffer
        return {(1 << (l - lp)) << w, 1 << w,
                (a + ((size_t)spad_size(1 << (l - 1), lp) << w)) * 8u};
    const size_t b = (size_t)spad_size(1 << l, lp) << w;
    return {(1 << (l - lp)) << w, 1 << w, std::max(a, b) * 8u};
}
Geo strided_geo(int l, int log2minw) {
    const int w = cols_log2w(l, log2minw);
    return {(1 << cols_log2t(l)) << w, 1 << w, padded_bytes(l, cols_maxrb(l), w)};
}
Geo real_geo(int lh) {
    const int w = real_log2w(lh), lp = sched_rbits(lh, real_maxrb(lh), 0);
    const int srow = sched_npass(lh, real_maxrb(lh)) > 1 ? spad_size(1 << lh, lp) : 0;
    const int slots = std::max(srow, (1 << lh) + 1);
    return {(1 << real_log2t(lh)) << w, 1 << w, (size_t)slots * (1u << w) * 8u};
}

std::string describe_spec(const PlanSpec& s, int64_t mmax, int real_pair = 0) {
    char buf[512];
    const char* dir = s.direction < 0 ? "forward" : "inverse";
    switch (s.path) {
        case PATH_ONEPASS: {
            Geo g = rows_geo(s.log2n);
            snprintf(buf, sizeof buf,
                     "path=onepass n=%lld batch=%lld %s shift=%d radix=%s kernels=1 "
                     "threads=%d rows_per_cta=%d smem=%zu",
                     (long long)s.n, (long long)s.batch, dir, s.shift,
                     radix_string(s.log2n, rows_maxrb(s.log2n)).c_str(), g.threads, g.per_cta, g.smem);
            break;
        }
        case PATH_FOURSTEP: {
            Geo g1 = cols_geo(s.log2n1, s.log2n2), g2 = rowst_geo(s.log2n2);
            snprintf(buf, sizeof buf,
                     "path=fourstep n=%lld batch=%lld %s shift=%d n1=%d n2=%d kernels=2 "
                     "pass1=columns(radix=%s threads=%d cols_per_cta=%d smem=%zu) "
                     "pass2=rows_transposed(radix=%s threads=%d rows_per_cta=%d smem=%zu)",
                     (long long)s.n, (long long)s.batch, dir, s.shift, 1 << s.log2n1,
                     1 << s.log2n2, radix_string(s.log2n1, cols_pass_maxrb(s.log2n1, s.log2n2)).c_str(), g1.threads,
                     g1.per_cta, g1.smem, radix_string(s.log2n2, rowst_maxrb(s.log2n2)).c_str(),
                     g2.threads, g2.per_cta, g2.smem);
            break;
        }
        case PATH_BLUESTEIN: {
            const bool light = blu_light(s.log2m, s.batch);
            const int w = blu_log2w(s.log2m, light);
            const bool real = s.layout != FFT_LAYOUT_C2C;
            char what[96];
            if (real)
                snprintf(what, sizeof what, "%s mmax=%lld layout=%s",
                         s.direction < 0 ? "analysis(r2c)" : "synthesis(c2r)", (long long)mmax,
                         s.layout == FFT_LAYOUT_REAL_MMAJOR ? "mmajor" : "rowmajor");
            else
                snprintf(what, sizeof what, "%s shift=%d", dir, s.shift);
            snprintf(buf, sizeof buf,
                     "path=bluestein n=%lld batch=%lld %s%s m=%d radix=%s kernels=1 "
                     "threads=%d rows_per_cta=%d smem=%zu",
                     (long long)s.n, (long long)s.batch, what,
                     real && real_pair ? " rows_per_transform=2" : "", 1 << s.log2m,
                     radix_string(s.log2m, blu_maxrb(s.log2m, light)).c_str(),
                     (1 << blu_log2t(s.log2m, light)) << w, 1 << w,
                     padded_bytes(s.log2m, blu_maxrb(s.log2m, light), w));
            break;
        }
        case PATH_MIXED: {
            const bool real = s.layout != FFT_LAYOUT_C2C;
            char what[96];
            if (real)
                snprintf(what, sizeof what, "%s mmax=%lld layout=%s",
                         s.direction < 0 ? "analysis(r2c)" : "synthesis(c2r)", (long long)mmax,
                         s.layout == FFT_LAYOUT_REAL_MMAJOR ? "mmajor" : "rowmajor");
            else
                snprintf(what, sizeof what, "%s shift=%d", dir, s.shift);
            std::string rs;
            for (int p = 0; p < s.nmix; ++p) rs += (p ? "x" : "") + std::to_string(s.mix_radix[p]);
            const int64_t ntr = real && real_pair ? (s.batch + 1) / 2 : s.batch;
            const bool small = mixed_small_cta((int)s.n, ntr);
            snprintf(buf, sizeof buf,
                     "path=mixed n=%lld batch=%lld %s%s radix=%s kernels=1 threads=%d "
                     "rows_per_cta=%d smem=%zu",
                     (long long)s.n, (long long)s.batch, what,
                     real && real_pair ? " rows_per_transform=2" : "", rs.c_str(),
                     mixed_threads_for(small), mixed_rows_for((int)s.n, small),
                     mixed_smem_bytes_for((int)s.n, small));
            break;
        }
        case PATH_MIXED_FS: {
            std::string r1, r2;
            for (int p = 0; p < s.nmix1; ++p) r1 += (p ? "x" : "") + std::to_string(s.mix_radix1[p]);
            for (int p = 0; p < s.nmix; ++p) r2 += (p ? "x" : "") + std::to_string(s.mix_radix[p]);
            const bool real = s.layout != FFT_LAYOUT_C2C;
            char what[128];
            if (real)
                snprintf(what, sizeof what, "%s mmax=%lld layout=%s rows_per_transform=2 kernels=%d",
                         s.direction < 0 ? "analysis(r2c)" : "synthesis(c2r)", (long long)mmax,
                         s.layout == FFT_LAYOUT_REAL_MMAJOR ? "mmajor" : "rowmajor",
                         s.direction < 0 ? 3 : 2);
            else
                snprintf(what, sizeof what, "%s shift=%d kernels=2", dir, s.shift);
            snprintf(buf, sizeof buf,
                     "path=mixed_fourstep n=%lld batch=%lld %s n1=%d n2=%d "
                     "pass1=columns(radix=%s cols_per_cta=%d smem=%zu) "
                     "pass2=rows_transposed(radix=%s rows_per_cta=%d smem=%zu)%s",
                     (long long)s.n, (long long)s.batch, what, s.mix_n1, s.mix_n2,
                     r1.c_str(), mixed_cols_per_cta(s.mix_n1), mixed_cols_smem_bytes(s.mix_n1),
                     r2.c_str(), mixed_rows_per_cta(s.mix_n2), mixed_smem_bytes(s.mix_n2),
                     real && s.direction < 0 ? " pass3=unpack" : "");
            break;
        }
        case PATH_BLUESTEIN_MP: {
            const bool real = s.layout != FFT_LAYOUT_C2C;
            char what[128];
            if (real)
                snprintf(what, sizeof what, "%s mmax=%lld layout=%s rows_per_transform=2",
                         s.direction < 0 ? "analysis(r2c)" : "synthesis(c2r)", (long long)mmax,
                         s.layout == FFT_LAYOUT_REAL_MMAJOR ? "mmajor" : "rowmajor");
            else
                snprintf(what, sizeof what, "%s shift=%d", dir, s.shift);
            snprintf(buf, sizeof buf,
                     "path=bluestein_multipass n=%lld batch=%lld %s m=%d n1=%d n2=%d kernels=6 "
                     "(chirp, fourstep fwd x2, fourstep inv x2 with the filter, chirp)",
                     (long long)s.n, (long long)s.batch, what, 1 << s.log2m, 1 << s.log2n1,
                     1 << s.log2n2);
            break;
        }
        case PATH_2D: {  // ny x n images: n-point rows, then ny-point columns
            Geo g1 = rows_geo(s.log2n), g2 = cols_geo(s.log2ny, s.log2n);
            snprintf(buf, sizeof buf,
                     "path=2d n=%lldx%lld batch=%lld %s shift=%d radix=%s kernels=2 "
                     "rows(threads=%d rows_per_cta=%d smem=%zu) "
                     "columns(radix=%s threads=%d cols_per_cta=%d smem=%zu)",
                     (long long)s.ny, (long long)s.n, (long long)s.batch, dir, s.shift,
                     radix_string(s.log2n, rows_maxrb(s.log2n)).c_str(), g1.threads, g1.per_cta,
                     g1.smem, radix_string(s.log2ny, cols_pass_maxrb(s.log2ny, s.log2n)).c_str(),
                     g2.threads, g2.per_cta, g2.smem);
            break;
        }
        default: {
            if (real_pair) {  // two rows per n-point complex transform
                const int l = s.log2n, w = rows_log2w(l), lp = sched_rbits(l, rows_maxrb(l), 0);
                const size_t slots = std::max(
                    (size_t)(sched_npass(l, rows_maxrb(l)) > 1 ? spad_size(1 << l, lp) : 0),
                    (size_t)1 << l);
                snprintf(buf, sizeof buf,
                         "path=real n=%lld batch=%lld %s mmax=%lld layout=%s core=%lld "
                         "rows_per_transform=2 radix=%s kernels=1 threads=%d pairs_per_cta=%d "
                         "smem=%zu",
                         (long long)s.n, (long long)s.batch,
                         s.direction < 0 ? "analysis(r2c)" : "synthesis(c2r)", (long long)mmax,
                         s.layout == FFT_LAYOUT_REAL_MMAJOR ? "mmajor" : "rowmajor",
                         (long long)s.n, radix_string(l, rows_maxrb(l)).c_str(),
                         (1 << rows_log2t(l)) << w, 1 << w, (slots << w) * 8u);
                break;
            }
            Geo g = real_geo(s.log2n - 1);
            snprintf(buf, sizeof buf,
                     "path=real n=%lld batch=%lld %s mmax=%lld layout=%s core=%lld radix=%s "
                     "kernels=1 threads=%d rows_per_cta=%d smem=%zu",
                     (long long)s.n, (long long)s.batch,
                     s.direction < 0 ? "analysis(r2c)" : "synthesis(c2r)", (long long)mmax,
                     s.layout == FFT_LAYOUT_REAL_MMAJOR ? "mmajor" : "rowmajor",
                     (long long)(s.n / 2), radix_string(s.log2n - 1, real_maxrb(s.log2n - 1)).c_str(), g.threads,
                     g.per_cta, g.smem);
            break;
        }
    }
    return buf;
}

// The chirp-z schedule of a plan, chosen from its batch (the tables follow the same choice).
int blu_mode_light(const PlanSpec& s) { return blu_light(s.log2m, s.batch) ? BLU_LIGHT : 0; }

int map_cuda(cudaError_t e) {
    if (e == cudaSuccess) return FFT_OK;
    return e == cudaErrorMemoryAllocation ? FFT_ERR_OOM : FFT_ERR_CUDA;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t a0 = (uintptr_t)a, b0 = (uintptr_t)b;
    return a0 < b0 + nb && b0 < a0 + na;
}

}  // namespace

struct gbfft_plan_s {
    PlanSpec s;
    int64_t mmax = 0;
    int device = 0;
    float2* d_tw = nullptr;
    size_t tw_count = 0;
    size_t off_a = 0, off_b = 0, off_hi = 0, off_lo = 0, off_r = 0;
    size_t off_pair = 0;  // real plans: pass tables of the n-point complex core (pairing)
    size_t off_chirp = 0, off_chirp_out = 0, off_bhat = 0;  // chirp-z tables
    void* d_work = nullptr;
    size_t work_bytes = 0;
    int* d_err = nullptr;
    uint64_t wait_limit_ns = 2000000000ull;  // bounded device waits: 2 s
    int normalize = 0;                       // 1: output scaled by 1/n (1/(nx*ny) for 2-D)
    int real_pair = 0;                       // 1: two real rows per complex transform
    int index_only = 0;                      // diagnostic: epilogues only (fft_plan_set_diagnostic)
    MixedSched mix = {};                     // mixed-radix schedule (offsets relative to off_a;
                                             // four-step: the N2 pass, relative to off_b)
    MixedSched mix1 = {};                    // four-step: the N1 pass (relative to off_a)
};

static void free_plan(gbfft_plan_s* p) {
    if (!p) return;
    if (p->d_tw) cudaFree(p->d_tw);
    if (p->d_work) cudaFree(p->d_work);
    if (p->d_err) cudaFree(p->d_err);
    delete p;
}

extern "C" {

int fft_version(void) { return 10000; }

const char* fft_status_string(int status) {
    switch (status) {
        case FFT_OK: return "FFT_OK: success";
        case FFT_ERR_INVALID_ARG: return "FFT_ERR_INVALID_ARG: invalid argument";
        case FFT_ERR_UNSUPPORTED_SIZE:
            return "FFT_ERR_UNSUPPORTED_SIZE: size outside the supported lengths";
        case FFT_ERR_MISALIGNED: return "FFT_ERR_MISALIGNED: data pointer not 16-byte aligned";
        case FFT_ERR_OOM: return "FFT_ERR_OOM: device allocation failed";
        case FFT_ERR_CUDA: return "FFT_ERR_CUDA: CUDA runtime or launch error";
        case FFT_ERR_TIMEOUT: return "FFT_ERR_TIMEOUT: a bounded device-side wait gave up";
        case FFT_ERR_BOUNDS:
            return "FFT_ERR_BOUNDS: a device index check of the checked build failed";
        default: return "unknown status";
    }
}

int fft_plan_query(int64_t n, int64_t batch, int dims, int direction, int layout, int shift,
                   char* buf, size_t len) {
    PlanSpec s;
    const int rc = plan_spec(n, batch, dims, direction, layout, shift, &s);
    if (rc != FFT_OK) return rc;
    if (buf && len) {
        std::string d = describe_spec(s, s.layout != FFT_LAYOUT_C2C ? (s.n - 1) / 2 : 0);
        snprintf(buf, len, "%s", d.c_str());
    }
    return FFT_OK;
}

static int create_from_spec(const PlanSpec& s, fft_plan* out);

int fft_plan_create(int64_t n, int64_t batch, int dims, int direction, int layout, int shift,
                    fft_plan* out) {
    if (!out) return FFT_ERR_INVALID_ARG;
    *out = nullptr;
    PlanSpec s;
    const int rc = plan_spec(n, batch, dims, direction, layout, shift, &s);
    return rc != FFT_OK ? rc : create_from_spec(s, out);
}

int fft_plan_create_2d(int64_t nx, int64_t ny, int64_t batch, int direction, int shift,
                       fft_plan* out) {
    if (!out) return FFT_ERR_INVALID_ARG;
    *out = nullptr;
    if (ny < 1) return FFT_ERR_UNSUPPORTED_SIZE;
    PlanSpec s;
    const int rc = plan_spec(nx, batch, 2, direction, FFT_LAYOUT_C2C, shift, &s, ny);
    return rc != FFT_OK ? rc : create_from_spec(s, out);
}

int fft_plan_query_2d(int64_t nx, int64_t ny, int64_t batch, int direction, int shift,
                      char* buf, size_t len) {
    if (ny < 1) return FFT_ERR_UNSUPPORTED_SIZE;
    PlanSpec s;
    const int rc = plan_spec(nx, batch, 2, direction, FFT_LAYOUT_C2C, shift, &s, ny);
    if (rc != FFT_OK) return rc;
    if (buf && len) snprintf(buf, len, "%s", describe_spec(s, 0).c_str());
    return FFT_OK;
}

static int create_from_spec(const PlanSpec& s, fft_plan* out) {

    gbfft_plan_s* p = new (std::nothrow) gbfft_plan_s();
    if (!p) return FFT_ERR_OOM;
    p->s = s;
    p->mmax = s.layout != FFT_LAYOUT_C2C ? (s.n - 1) / 2 : 0;  // largest m with 2m < n
    if (cudaGetDevice(&p->device) != cudaSuccess) {
        delete p;
        return FFT_ERR_CUDA;
    }

    std::vector<float2> tw;
    switch (s.path) {
        case PATH_ONEPASS:
            p->off_a = append_pass_tables(tw, s.log2n, rows_maxrb(s.log2n));
            break;
        case PATH_2D:
            p->off_a = append_pass_tables(tw, s.log2n, rows_maxrb(s.log2n));  // row pass
            p->off_b = append_pass_tables(tw, s.log2ny, cols_pass_maxrb(s.log2ny, s.log2n));
            break;
        case PATH_FOURSTEP: {
            p->off_a = append_pass_tables(tw, s.log2n1, cols_pass_maxrb(s.log2n1, s.log2n2));
            p->off_b = append_pass_tables(tw, s.log2n2, rowst_maxrb(s.log2n2));
            const int64_t nlo = int64_t(1) << s.lowbits, nhi = int64_t(1) << (s.log2n - s.lowbits);
            p->off_hi = append_roots(tw, nhi, nlo, s.n);  // w_n^{qh * 2^lowbits}
            p->off_lo = append_roots(tw, nlo, 1, s.n);    // w_n^{ql}
            p->work_bytes = (size_t)s.batch * (size_t)s.n * sizeof(float2);
            break;
        }
        case PATH_BLUESTEIN:
            p->off_a = append_pass_tables(tw, s.log2m, blu_maxrb(s.log2m, blu_light(s.log2m, s.batch)));
            {
                // fftshift folded in: exp(+2 pi i j h/n) on the forward load, exp(-2 pi i k h/n)
                // on the inverse store, h = n/2 rounded down
                const int64_t h = s.n / 2;
                const bool fwd = s.direction == FFT_FORWARD;
                p->off_chirp = host::append_chirp(tw, s.n, s.direction, s.shift && fwd ? h : 0);
                // a table of its own, so that fft_plan_set_normalization can rescale it
                p->off_chirp_out = host::append_chirp(tw, s.n, s.direction, s.shift && !fwd ? -h : 0);
            }
            p->off_bhat = host::append_chirp_filter(tw, s.n, int64_t(1) << s.log2m, s.direction);
            break;
        case PATH_MIXED_FS: {
            p->off_a = host::append_mixed_tables(tw, s.nmix1, s.mix_radix1, &p->mix1);
            p->off_b = host::append_mixed_tables(tw, s.nmix, s.mix_radix, &p->mix);
            const int64_t nlo = int64_t(1) << kMixedTwLoBits;
            p->off_lo = host::append_roots_any(tw, nlo, 1, s.n);                  // w_n^{ql}
            p->off_hi = host::append_roots_any(tw, (s.n + nlo - 1) / nlo, nlo, s.n);  // w_n^{qh*nlo}
            if (s.shift) p->off_chirp = host::append_phase(tw, s.n, s.n / 2);
            // complex rows: one workspace; real rows (two per transform): the column pass's
            // output and, for the analysis, the row pass's spectra before the unpack
            const int64_t ntr = s.layout == FFT_LAYOUT_C2C ? s.batch : 2 * ((s.batch + 1) / 2);
            p->work_bytes = (size_t)ntr * (size_t)s.n * sizeof(float2);
            break;
        }
        case PATH_MIXED: {
            p->off_a = host::append_mixed_tables(tw, s.nmix, s.mix_radix, &p->mix);
            if (s.shift)  // (cos, sin)(2*pi*(j*h mod n)/n), h = floor(n/2)
                p->off_chirp = host::append_phase(tw, s.n, s.n / 2);
            break;
        }
        case PATH_BLUESTEIN_MP: {
            p->off_a = append_pass_tables(tw, s.log2n1, cols_pass_maxrb(s.log2n1, s.log2n2));
            p->off_b = append_pass_tables(tw, s.log2n2, rowst_maxrb(s.log2n2));
            const int64_t m = int64_t(1) << s.log2m;
            const int64_t nlo = int64_t(1) << s.lowbits, nhi = int64_t(1) << (s.log2m - s.lowbits);
            p->off_hi = append_roots(tw, nhi, nlo, m);  // w_m^{qh * 2^lowbits}
            p->off_lo = append_roots(tw, nlo, 1, m);    // w_m^{ql}
            const int64_t h = s.n / 2;
            const bool fwd = s.direction == FFT_FORWARD;
            const bool c2c = s.layout == FFT_LAYOUT_C2C;
            p->off_chirp = host::append_chirp(tw, s.n, s.direction, c2c && s.shift && fwd ? h : 0);
            p->off_chirp_out =
                host::append_chirp(tw, s.n, s.direction, c2c && s.shift && !fwd ? -h : 0);
            p->off_bhat = host::append_chirp_filter(tw, s.n, m, s.direction);
            const int64_t ntr = c2c ? s.batch : (s.batch + 1) / 2;
            p->work_bytes = 2 * (size_t)ntr * (size_t)m * sizeof(float2);  // A and B
            break;
        }
        case PATH_REAL:
            p->off_a = append_pass_tables(tw, s.log2n - 1, real_maxrb(s.log2n - 1));
            p->off_r = append_roots(tw, s.n / 2, 1, s.n);  // w_n^k, k < n/2
            if (s.log2n <= kMaxLog2RealPair)  // n-point core of the two-rows-per-transform option
                p->off_pair = append_pass_tables(tw, s.log2n, rows_maxrb(s.log2n));
            break;
    }
    align_table(tw);
    if (tw.empty()) tw.resize(32, make_float2(0.f, 0.f));
    p->tw_count = tw.size();

    cudaError_t e = cudaMalloc((void**)&p->d_tw, tw.size() * sizeof(float2));
    if (e == cudaSuccess)
        e = cudaMemcpy(p->d_tw, tw.data(), tw.size() * sizeof(float2), cudaMemcpyHostToDevice);
    if (e == cudaSuccess) e = cudaMalloc((void**)&p->d_err, sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(p->d_err, 0, sizeof(int));
    if (e == cudaSuccess && p->work_bytes) e = cudaMalloc(&p->d_work, p->work_bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error state of a failed allocation
        free_plan(p);
        return map_cuda(e);
    }
    *out = p;
    return FFT_OK;
}

int fft_plan_set_normalization(fft_plan p, int normalize) {
    if (!p || p->s.layout != FFT_LAYOUT_C2C || (normalize != 0 && normalize != 1))
        return FFT_ERR_INVALID_ARG;
    const PlanSpec& s = p->s;
    if ((s.path == PATH_BLUESTEIN || s.path == PATH_BLUESTEIN_MP) && normalize != p->normalize) {
        // the chirp of the store, times 1/n when normalising (rewritten in place)
        std::vector<float2> t;
        const bool fwd = s.direction == FFT_FORWARD;
        const size_t off = host::append_chirp(t, s.n, s.direction, s.shift && !fwd ? -(s.n / 2) : 0);
        const float f = normalize ? (float)(1.0 / (double)s.n) : 1.f;
        for (size_t i = off; i < t.size(); ++i) t[i] = make_float2(t[i].x * f, t[i].y * f);
        if (cudaMemcpy(p->d_tw + p->off_chirp_out, t.data() + off,
                       (t.size() - off) * sizeof(float2), cudaMemcpyHostToDevice) != cudaSuccess)
            return FFT_ERR_CUDA;
    }
    p->normalize = normalize;
    return FFT_OK;
}

int fft_plan_set_band_limit(fft_plan p, int64_t mmax) {
    if (!p || p->s.layout == FFT_LAYOUT_C2C) return FFT_ERR_INVALID_ARG;
    if (mmax < 0 || 2 * mmax > p->s.n) return FFT_ERR_INVALID_ARG;  // mmax = n/2: Nyquist
    p->mmax = mmax;
    return FFT_OK;
}

int fft_plan_set_real_pairing(fft_plan p, int pairing) {
    if (!p || p->s.layout == FFT_LAYOUT_C2C || (pairing != 0 && pairing != 1))
        return FFT_ERR_INVALID_ARG;
    if (pairing && p->s.path == PATH_REAL && p->s.log2n > kMaxLog2RealPair)
        return FFT_ERR_UNSUPPORTED_SIZE;
    p->real_pair = pairing;
    return FFT_OK;
}

// The (path, size) combinations whose kernels carry the index-only diagnostic.
static bool index_only_supported(const gbfft_plan_s* p) {
    const PlanSpec& s = p->s;
    switch (s.path) {
        case PATH_ONEPASS: return s.log2n == 12;
        case PATH_FOURSTEP: return s.log2n == 15;
        case PATH_REAL: return p->real_pair ? s.log2n == 12 : (s.log2n == 12 || s.log2n == 15);
        default: return false;
    }
}

int fft_plan_set_diagnostic(fft_plan p, int mode) {
    if (!p || (mode != 0 && mode != FFT_DIAG_INDEX_ONLY)) return FFT_ERR_INVALID_ARG;
    p->index_only = mode == FFT_DIAG_INDEX_ONLY;
    if (p->index_only && !index_only_supported(p)) {
        p->index_only = 0;
        return FFT_ERR_UNSUPPORTED_SIZE;
    }
    return FFT_OK;
}

int fft_plan_set_wait_timeout(fft_plan p, uint64_t ns) {
    if (!p) return FFT_ERR_INVALID_ARG;
    p->wait_limit_ns = ns;
    return FFT_OK;
}

int fft_plan_workspace_bytes(fft_plan p, size_t* bytes) {
    if (!p || !bytes) return FFT_ERR_INVALID_ARG;
    *bytes = p->work_bytes;
    return FFT_OK;
}

int fft_plan_describe(fft_plan p, char* buf, size_t len) {
    if (!p || !buf || !len) return FFT_ERR_INVALID_ARG;
    std::string d = describe_spec(p->s, p->mmax, p->real_pair);
    snprintf(buf, len, "%s", d.c_str());
    return FFT_OK;
}

static cudaError_t exec_chirp_mp(fft_plan p, int mode, const void* in, void* out,
                                 cudaStream_t st) {
    const PlanSpec& s = p->s;
    ChirpMpTables t;
    t.chirp = p->d_tw + p->off_chirp;
    t.chirp_out = p->d_tw + p->off_chirp_out;
    t.bhat = p->d_tw + p->off_bhat;
    t.tw_cols = p->d_tw + p->off_a;
    t.tw_rows = p->d_tw + p->off_b;
    t.hi = p->d_tw + p->off_hi;
    t.lo = p->d_tw + p->off_lo;
    t.lowbits = s.lowbits;
    float2* A = (float2*)p->d_work;
    float2* B = A + p->work_bytes / (2 * sizeof(float2));
    return run_bluestein_mp(mode, in, out, s.batch, (int)s.n, s.log2m, (int)p->mmax,
                            s.layout == FFT_LAYOUT_REAL_MMAJOR, t, A, B, p->d_err,
                            p->wait_limit_ns, st);
}

int fft_exec_c2c(fft_plan p, const void* in, void* out, void* stream) {
    if (!p || !in || !out) return FFT_ERR_INVALID_ARG;
    const PlanSpec& s = p->s;
    if (s.layout != FFT_LAYOUT_C2C) return FFT_ERR_INVALID_ARG;
    if (!aligned16(in) || !aligned16(out)) return FFT_ERR_MISALIGNED;
    const size_t bytes = (size_t)s.batch * (size_t)(s.dims == 2 ? s.n * s.ny : s.n) * 8u;
    if (in != out && ranges_overlap(in, bytes, out, bytes)) return FFT_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    const float2* x = (const float2*)in;
    float2* y = (float2*)out;
    const bool fwd = s.direction == FFT_FORWARD;
    if (p->index_only && !index_only_supported(p)) return FFT_ERR_UNSUPPORTED_SIZE;
    const int diag = p->index_only ? KF_INDEX_ONLY : 0;
    cudaError_t e = cudaSuccess;
    switch (s.path) {
        case PATH_ONEPASS: {
            const int flags = (s.shift ? (fwd ? KF_CHESS_LOAD : KF_CHESS_STORE) : 0) |
                              (p->normalize ? kf_scale(s.log2n) : 0) | diag;
            e = run_rows(s.log2n, s.direction, x, y, s.batch, p->d_tw + p->off_a, flags, 0,
                         p->d_err, p->wait_limit_ns, st);
            break;
        }
        case PATH_BLUESTEIN: {  // the shift lives in the chirp tables
            e = run_bluestein(s.log2m, BLU_C2C | blu_mode_light(s), x, y, s.batch, (int)s.n, 0, 0,
                              p->d_tw + p->off_chirp,
                              p->d_tw + p->off_chirp_out, p->d_tw + p->off_bhat,
                              p->d_tw + p->off_a, st);
            break;
        }
        case PATH_MIXED_FS: {  // in == out is fine: pass 1 writes only the workspace
            float2* wk = (float2*)p->d_work;
            e = run_mixed_cols(s.direction, x, wk, s.batch, s.mix_n1, s.mix_n2, p->mix1,
                               p->d_tw + p->off_a, p->d_tw + p->off_hi, p->d_tw + p->off_lo,
                               kMixedTwLoBits, p->d_tw + p->off_chirp, s.shift && fwd, st);
            if (e == cudaSuccess)
                e = run_mixed(kMixedRowsT, s.direction, wk, y, s.batch * s.mix_n1, s.mix_n2,
                              p->mix, p->d_tw + p->off_b, p->d_tw + p->off_chirp, 0,
                              s.shift && !fwd, p->normalize ? (float)(1.0 / (double)s.n) : 1.f,
                              0, 0, st, s.mix_n1);
            break;
        }
        case PATH_MIXED:  // in == out is fine: each CTA reads its rows before writing them
            e = run_mixed(BLU_C2C, s.direction, x, y, s.batch, (int)s.n, p->mix,
                          p->d_tw + p->off_a, p->d_tw + p->off_chirp, s.shift && fwd,
                          s.shift && !fwd, p->normalize ? (float)(1.0 / (double)s.n) : 1.f, 0, 0,
                          st);
            break;
        case PATH_BLUESTEIN_MP:  // in == out is fine: the input is read into the workspace first
            e = exec_chirp_mp(p, 0, x, y, st);
            break;
        case PATH_FOURSTEP: {
            float2* wk = (float2*)p->d_work;
            const int64_t n1 = int64_t(1) << s.log2n1, n2 = int64_t(1) << s.log2n2;
            e = run_cols(s.log2n1, s.direction, x, wk, s.batch * n2, s.log2n2,
                         p->d_tw + p->off_a, ((s.shift && fwd) ? KF_CHESS_LOAD : 0) | diag, 0,
                         p->d_tw + p->off_hi, p->d_tw + p->off_lo, s.lowbits, p->d_err,
                         p->wait_limit_ns, st);
            if (e == cudaSuccess)
                e = run_rows_t(s.log2n2, s.direction, wk, y, s.batch * n1, s.log2n1,
                               p->d_tw + p->off_b,
                               ((s.shift && !fwd) ? KF_CHESS_STORE : 0) |
                                   (p->normalize ? kf_scale(s.log2n) : 0) | diag,
                               p->d_err, p->wait_limit_ns, st);
            break;
        }
        case PATH_2D: {  // batch*ny rows of n points, then batch*n columns of ny points
            e = run_rows(s.log2n, s.direction, x, y, s.batch * s.ny, p->d_tw + p->off_a,
                         (s.shift && fwd) ? KF_CHESS_LOAD : 0, 1, p->d_err, p->wait_limit_ns, st);
            if (e == cudaSuccess)
                e = run_cols(s.log2ny, s.direction, y, y, s.batch * s.n, s.log2n,
                             p->d_tw + p->off_b,
                             ((s.shift && !fwd) ? KF_CHESS_STORE : 0) |
                                 (p->normalize ? kf_scale(s.log2n + s.log2ny) : 0),
                             1, nullptr, nullptr, 0, p->d_err, p->wait_limit_ns, st);
            break;
        }
        default:
            return FFT_ERR_INVALID_ARG;
    }
    return e == cudaSuccess ? FFT_OK : FFT_ERR_CUDA;
}

int fft_exec_r2c(fft_plan p, const float* in, void* out, void* stream) {
    if (!p || !in || !out) return FFT_ERR_INVALID_ARG;
    const PlanSpec& s = p->s;
    if (s.layout == FFT_LAYOUT_C2C || s.direction != FFT_FORWARD) return FFT_ERR_INVALID_ARG;
    if (!aligned16(in) || !aligned16(out)) return FFT_ERR_MISALIGNED;
    const size_t in_bytes = (size_t)s.batch * (size_t)s.n * 4u;
    const size_t out_bytes = (size_t)s.batch * (size_t)(p->mmax + 1) * 8u;
    if (ranges_overlap(in, in_bytes, out, out_bytes)) return FFT_ERR_INVALID_ARG;
    const int mmajor = s.layout == FFT_LAYOUT_REAL_MMAJOR;
    if (p->index_only && !index_only_supported(p)) return FFT_ERR_UNSUPPORTED_SIZE;
    const int diag = p->index_only ? KF_INDEX_ONLY : 0;
    cudaError_t e;
    if (s.path == PATH_MIXED_FS) {  // pack, columns; rows; unpack
        const cudaStream_t st = (cudaStream_t)stream;
        const int64_t ntr = (s.batch + 1) / 2;
        float2* A = (float2*)p->d_work;
        float2* B = A + ntr * s.n;
        e = run_mixed_cols_real(BLU_R2C2, in, A, s.batch, s.mix_n1, s.mix_n2, p->mix1,
                                p->d_tw + p->off_a, p->d_tw + p->off_hi, p->d_tw + p->off_lo,
                                kMixedTwLoBits, (int)p->mmax, mmajor, st);
        if (e == cudaSuccess)
            e = run_mixed(kMixedRowsT, -1, A, B, ntr * s.mix_n1, s.mix_n2, p->mix,
                          p->d_tw + p->off_b, p->d_tw, 0, 0, 1.f, 0, 0, st, s.mix_n1);
        if (e == cudaSuccess)
            e = run_mixed_unpack(B, (float2*)out, s.batch, (int)s.n, (int)p->mmax, mmajor, st);
    } else if (s.path == PATH_MIXED)
        e = run_mixed(p->real_pair ? BLU_R2C2 : BLU_R2C, -1, in, out, s.batch, (int)s.n, p->mix,
                      p->d_tw + p->off_a, nullptr, 0, 0, 1.f, (int)p->mmax, mmajor,
                      (cudaStream_t)stream);
    else if (s.path == PATH_BLUESTEIN_MP)
        e = exec_chirp_mp(p, 3, in, out, (cudaStream_t)stream);
    else if (s.path == PATH_BLUESTEIN)
        e = run_bluestein(s.log2m, (p->real_pair ? BLU_R2C2 : BLU_R2C) | blu_mode_light(s), in, out,
                          s.batch, (int)s.n,
                          (int)p->mmax, mmajor, p->d_tw + p->off_chirp, p->d_tw + p->off_chirp_out,
                          p->d_tw + p->off_bhat, p->d_tw + p->off_a, (cudaStream_t)stream);
    else if (p->real_pair)
        e = run_real_pair(s.log2n, true, in, out, s.batch, (int)p->mmax, mmajor,
                          p->d_tw + p->off_pair, diag, (cudaStream_t)stream);
    else
        e = run_r2c(s.log2n - 1, in, (float2*)out, s.batch, (int)p->mmax, mmajor,
                    p->d_tw + p->off_a, p->d_tw + p->off_r, diag, p->d_err, p->wait_limit_ns,
                    (cudaStream_t)stream);
    return e == cudaSuccess ? FFT_OK : FFT_ERR_CUDA;
}

int fft_exec_c2r(fft_plan p, const void* in, float* out, void* stream) {
    if (!p || !in || !out) return FFT_ERR_INVALID_ARG;
    const PlanSpec& s = p->s;
    if (s.layout == FFT_LAYOUT_C2C || s.direction != FFT_INVERSE) return FFT_ERR_INVALID_ARG;
    if (!aligned16(in) || !aligned16(out)) return FFT_ERR_MISALIGNED;
    const size_t in_bytes = (size_t)s.batch * (size_t)(p->mmax + 1) * 8u;
    const size_t out_bytes = (size_t)s.batch * (size_t)s.n * 4u;
    if (ranges_overlap(in, in_bytes, out, out_bytes)) return FFT_ERR_INVALID_ARG;
    const int mmajor = s.layout == FFT_LAYOUT_REAL_MMAJOR;
    if (p->index_only && !index_only_supported(p)) return FFT_ERR_UNSUPPORTED_SIZE;
    const int diag = p->index_only ? KF_INDEX_ONLY : 0;
    cudaError_t e;
    if (s.path == PATH_MIXED_FS) {  // assemble, columns; rows split into the real rows
        const cudaStream_t st = (cudaStream_t)stream;
        float2* A = (float2*)p->d_work;
        e = run_mixed_cols_real(BLU_C2R2, in, A, s.batch, s.mix_n1, s.mix_n2, p->mix1,
                                p->d_tw + p->off_a, p->d_tw + p->off_hi, p->d_tw + p->off_lo,
                                kMixedTwLoBits, (int)p->mmax, mmajor, st);
        if (e == cudaSuccess)
            e = run_mixed_rows_split(A, out, s.batch, s.mix_n1, s.mix_n2, p->mix,
                                     p->d_tw + p->off_b, st);
    } else if (s.path == PATH_MIXED)
        e = run_mixed(p->real_pair ? BLU_C2R2 : BLU_C2R, +1, in, out, s.batch, (int)s.n, p->mix,
                      p->d_tw + p->off_a, nullptr, 0, 0, 1.f, (int)p->mmax, mmajor,
                      (cudaStream_t)stream);
    else if (s.path == PATH_BLUESTEIN_MP)
        e = exec_chirp_mp(p, 4, in, out, (cudaStream_t)stream);
    else if (s.path == PATH_BLUESTEIN)
        e = run_bluestein(s.log2m, (p->real_pair ? BLU_C2R2 : BLU_C2R) | blu_mode_light(s), in, out,
                          s.batch, (int)s.n,
                          (int)p->mmax, mmajor, p->d_tw + p->off_chirp, p->d_tw + p->off_chirp_out,
                          p->d_tw + p->off_bhat, p->d_tw + p->off_a, (cudaStream_t)stream);
    else if (p->real_pair)
        e = run_real_pair(s.log2n, false, in, out, s.batch, (int)p->mmax, mmajor,
                          p->d_tw + p->off_pair, diag, (cudaStream_t)stream);
    else
        e = run_c2r(s.log2n - 1, (const float2*)in, out, s.batch, (int)p->mmax, mmajor,
                    p->d_tw + p->off_a, p->d_tw + p->off_r, diag, p->d_err, p->wait_limit_ns,
                    (cudaStream_t)stream);
    return e == cudaSuccess ? FFT_OK : FFT_ERR_CUDA;
}

int fft_plan_check(fft_plan p) {
    if (!p) return FFT_ERR_INVALID_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess) return FFT_ERR_CUDA;
    int h = 0;
    if (cudaMemcpy(&h, p->d_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return FFT_ERR_CUDA;
    if (h != 0) {
        if (cudaMemset(p->d_err, 0, sizeof(int)) != cudaSuccess) return FFT_ERR_CUDA;
        return kerr_status(h);
    }
    return FFT_OK;
}

int fft_plan_destroy(fft_plan p) {
    if (!p) return FFT_OK;
    const cudaError_t e = cudaDeviceSynchronize();
    free_plan(p);
    return e == cudaSuccess ? FFT_OK : FFT_ERR_CUDA;
}

}  // extern "C"
