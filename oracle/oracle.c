/*
 * fp64 CPU oracle for the batched FFT library.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is compiled into oracle/liboracle.so and is called
 * from tests/, from __graft_entry__.smoke() and from the CPU-baseline leg of bench.py.  It is
 * never linked into, imported by, or called from the CUDA library, and it shares no code,
 * header, table or constant with it.  It is deliberately plain and slow: every function is
 * the textbook definition (or the textbook recursive radix-2 FFT) written out in double
 * precision so that a reader can check it against the pages by eye.
 *
 * Sources (page title, then the section / equation used):
 *   [Mota]   "High Performance Fourier Transforms on GPUs with GLSL" (MSc dissertation,
 *            U. Minho, 2023): §2.2 Eq. 5 (DFT definition), §2.3.1 Eq. 9-10 (radix-2
 *            decimation-in-time split and butterfly), §2.7 Eq. 19 (2-D row-column).
 *   [SHT]    "src/sht/wgsl/fourier.ts" (WGSL Fourier-stage kernels of a spherical-harmonic
 *            transform): header comment (band-limited real synthesis / analysis, mmax < nphi/2),
 *            fftSynthWGSL (Hermitian assembly X_0 = Re F_0, X_m = F_m, X_{N-m} = conj F_m),
 *            fftAnalysWGSL (keep m = 0..mmax), dftSynthWGSL / dftAnalysWGSL (direct
 *            band-limited sums, "also useful as a cross-check").
 *   [Shift]  "The 1D fftshift in CUDA by chessboard multiplication": "What is fftshift?"
 *            (zero frequency moved to the centre, i.e. a rotation by N/2 for even N).
 *
 * Conventions fixed here (readings of the pages):
 *   - X_k = sum_j x_j exp(s * 2*pi*i * j*k / N), s = -1 forward, s = +1 inverse, no 1/N
 *     scaling in either direction (the WGSL page's "Unnormalized" Stockham; Mota's Eq. 5
 *     divides the inverse by N, which this library does not do).
 *   - Complex data are interleaved (re, im) doubles; rows of a batch are contiguous.
 *   - Every exp(s*2*pi*i*q/N) is evaluated as cos/sin of 2*pi*(q mod N)/N in double, with the
 *     reduction q mod N done in exact integer arithmetic.
 *
 * Every entry point returns 0 on success and -1 on a bad argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    double re, im;
} cplx;

static const double kTwoPi = 6.283185307179586476925286766559005768;

static int is_pow2(int64_t n) { return n >= 1 && (n & (n - 1)) == 0; }

/* exp(s * 2*pi*i * q / n), q reduced mod n exactly. */
static cplx unit_root(int sign, int64_t q, int64_t n) {
    q %= n;
    if (q < 0) q += n;
    double th = kTwoPi * (double)q / (double)n;
    cplx w = {cos(th), (double)sign * sin(th)};
    return w;
}

static cplx cmul(cplx a, cplx b) {
    cplx r = {a.re * b.re - a.im * b.im, a.re * b.im + a.im * b.re};
    return r;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int t) {
#ifdef _OPENMP
    if (t >= 1) omp_set_num_threads(t);
#else
    (void)t;
#endif
}

/* ---------------------------------------------------------------------------------------
 * Direct DFT, [Mota] §2.2 Eq. 5: X_k = sum_{j<N} x_j w^{jk}, O(N^2) per row.
 * Any N >= 1 (not only powers of two).
 * ------------------------------------------------------------------------------------- */
int oracle_dft(const double* x, int64_t n, int64_t batch, int sign, double* out) {
    if (!x || !out || n < 1 || batch < 1 || (sign != 1 && sign != -1)) return -1;
    /* table w^q for q < n: the exponent j*k is reduced mod n before lookup */
    cplx* w = (cplx*)malloc(sizeof(cplx) * (size_t)n);
    if (!w) return -1;
    for (int64_t q = 0; q < n; ++q) w[q] = unit_root(sign, q, n);
#pragma omp parallel for schedule(dynamic)
    for (int64_t b = 0; b < batch; ++b) {
        const cplx* xr = (const cplx*)x + b * n;
        cplx* yr = (cplx*)out + b * n;
        for (int64_t k = 0; k < n; ++k) {
            double sre = 0.0, sim = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                int64_t q = (int64_t)(((__int128)j * k) % n);
                cplx t = cmul(xr[j], w[q]);
                sre += t.re;
                sim += t.im;
            }
            yr[k].re = sre;
            yr[k].im = sim;
        }
    }
    free(w);
    return 0;
}

/* Selected bins of one row, each by the direct sum of Eq. 5 (O(N) per bin). Used to check
 * sampled outputs of very large transforms one by one. */
int oracle_dft_bins(const double* x, int64_t n, int sign, const int64_t* bins, int64_t nbins,
                    double* out) {
    if (!x || !bins || !out || n < 1 || nbins < 0 || (sign != 1 && sign != -1)) return -1;
    const cplx* xr = (const cplx*)x;
#pragma omp parallel for schedule(dynamic)
    for (int64_t i = 0; i < nbins; ++i) {
        int64_t k = bins[i] % n;
        if (k < 0) k += n;
        double sre = 0.0, sim = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            int64_t q = (int64_t)(((__int128)j * k) % n);
            cplx t = cmul(xr[j], unit_root(sign, q, n));
            sre += t.re;
            sim += t.im;
        }
        out[2 * i] = sre;
        out[2 * i + 1] = sim;
    }
    return 0;
}

/* ---------------------------------------------------------------------------------------
 * Recursive radix-2 decimation-in-time FFT, [Mota] §2.3.1 Eq. 9-10:
 *   X_k       = E_k + w_N^k O_k
 *   X_{k+N/2} = E_k - w_N^k O_k,   k < N/2,
 * where E and O are the N/2-point DFTs of the even- and odd-indexed samples.
 * x is read with a stride (the even/odd split), out is written contiguously.
 * roots[q] = w_Ntop^q for q < Ntop/2, and an n-point level uses roots[k * (Ntop/n)].
 * ------------------------------------------------------------------------------------- */
static void fft_rec(const cplx* x, int64_t stride, int64_t n, const cplx* roots,
                    int64_t root_step, cplx* out) {
    if (n == 1) {
        out[0] = x[0];
        return;
    }
    int64_t h = n / 2;
    fft_rec(x, 2 * stride, h, roots, 2 * root_step, out);            /* E -> out[0, h)  */
    fft_rec(x + stride, 2 * stride, h, roots, 2 * root_step, out + h); /* O -> out[h, n) */
    for (int64_t k = 0; k < h; ++k) {
        cplx e = out[k];
        cplx t = cmul(roots[k * root_step], out[k + h]);
        out[k].re = e.re + t.re;
        out[k].im = e.im + t.im;
        out[k + h].re = e.re - t.re;
        out[k + h].im = e.im - t.im;
    }
}

static cplx* make_roots(int sign, int64_t n) {
    int64_t h = n / 2 > 0 ? n / 2 : 1;
    cplx* r = (cplx*)malloc(sizeof(cplx) * (size_t)h);
    if (!r) return NULL;
    for (int64_t q = 0; q < h; ++q) r[q] = unit_root(sign, q, n);
    return r;
}

/* Batched 1-D transform of contiguous rows (power-of-two n). out may equal x only if the
 * caller accepts a copy (handled here with a per-row temporary). */
int oracle_fft(const double* x, int64_t n, int64_t batch, int sign, double* out) {
    if (!x || !out || !is_pow2(n) || batch < 1 || (sign != 1 && sign != -1)) return -1;
    cplx* roots = make_roots(sign, n);
    if (!roots) return -1;
    int failed = 0;
#pragma omp parallel
    {
        cplx* tmp = (cplx*)malloc(sizeof(cplx) * (size_t)n);
        if (!tmp) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic)
            for (int64_t b = 0; b < batch; ++b) {
                fft_rec((const cplx*)x + b * n, 1, n, roots, 1, tmp);
                memcpy((cplx*)out + b * n, tmp, sizeof(cplx) * (size_t)n);
            }
            free(tmp);
        }
    }
    free(roots);
    return failed ? -1 : 0;
}

/* ---------------------------------------------------------------------------------------
 * 2-D transform of n x n images by row-column decomposition, [Mota] §2.7 Eq. 19:
 * 1-D transforms of every row, then of every column.
 * ------------------------------------------------------------------------------------- */
int oracle_fft2d(const double* x, int64_t n, int64_t batch, int sign, double* out) {
    if (!x || !out || !is_pow2(n) || batch < 1 || (sign != 1 && sign != -1)) return -1;
    if (oracle_fft(x, n, batch * n, sign, out) != 0) return -1; /* horizontal pass */
    cplx* roots = make_roots(sign, n);
    if (!roots) return -1;
    int failed = 0;
#pragma omp parallel
    {
        cplx* col = (cplx*)malloc(sizeof(cplx) * (size_t)n);
        cplx* res = (cplx*)malloc(sizeof(cplx) * (size_t)n);
        if (!col || !res) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic)
            for (int64_t bc = 0; bc < batch * n; ++bc) { /* vertical pass */
                int64_t b = bc / n, c = bc % n;
                cplx* img = (cplx*)out + b * n * n;
                for (int64_t r = 0; r < n; ++r) col[r] = img[r * n + c];
                fft_rec(col, 1, n, roots, 1, res);
                for (int64_t r = 0; r < n; ++r) img[r * n + c] = res[r];
            }
        }
        free(col);
        free(res);
    }
    free(roots);
    return failed ? -1 : 0;
}

/* ---------------------------------------------------------------------------------------
 * Mixed-radix recursive decimation in time for any N >= 1: [Mota] §2.3.1 Eq. 9-10 with the
 * radix p the smallest prime factor of N instead of 2,
 *   X_k = sum_{r<p} w_N^{r*k} Y_r[k mod N/p],   Y_r = the N/p-point DFT of x_r, x_{r+p}, ...,
 * and the direct sum of Eq. 5 when N itself is prime.  O(N * sum of the prime factors).
 * ------------------------------------------------------------------------------------- */
static int64_t smallest_prime_factor(int64_t n) {
    if (n % 2 == 0) return 2;
    for (int64_t p = 3; p * p <= n; p += 2)
        if (n % p == 0) return p;
    return n;
}

static int fft_any_rec(const cplx* x, int64_t stride, int64_t n, int sign, cplx* out) {
    if (n == 1) {
        out[0] = x[0];
        return 0;
    }
    const int64_t p = smallest_prime_factor(n), m = n / p;
    cplx* w = (cplx*)malloc(sizeof(cplx) * (size_t)n);  /* w_n^q, q < n */
    cplx* sub = (cplx*)malloc(sizeof(cplx) * (size_t)n); /* p transforms of m points */
    if (!w || !sub) {
        free(w);
        free(sub);
        return -1;
    }
    for (int64_t q = 0; q < n; ++q) w[q] = unit_root(sign, q, n);
    int rc = 0;
    if (p == n) { /* prime: the direct sum */
        for (int64_t j = 0; j < n; ++j) sub[j] = x[j * stride];
    } else {
        for (int64_t r = 0; r < p && rc == 0; ++r)
            rc = fft_any_rec(x + r * stride, stride * p, m, sign, sub + r * m);
    }
    for (int64_t k = 0; k < n && rc == 0; ++k) {
        double sre = 0.0, sim = 0.0;
        for (int64_t r = 0; r < p; ++r) {
            const cplx y = p == n ? sub[r] : sub[r * m + k % m];
            const cplx t = cmul(y, w[(int64_t)(((__int128)r * k) % n)]);
            sre += t.re;
            sim += t.im;
        }
        out[k].re = sre;
        out[k].im = sim;
    }
    free(w);
    free(sub);
    return rc;
}

int oracle_fft_any(const double* x, int64_t n, int64_t batch, int sign, double* out) {
    if (!x || !out || n < 1 || batch < 1 || (sign != 1 && sign != -1)) return -1;
    int failed = 0;
#pragma omp parallel for schedule(dynamic)
    for (int64_t b = 0; b < batch; ++b) {
        if (fft_any_rec((const cplx*)x + b * n, 1, n, sign, (cplx*)out + b * n) != 0) {
#pragma omp atomic write
            failed = 1;
        }
    }
    return failed ? -1 : 0;
}

/* ---------------------------------------------------------------------------------------
 * fftshift by index rotation, [Shift] "What is fftshift?": bin 0 moves to index N/2.
 * For even N the rotation by N/2 is its own inverse, so this is also ifftshift.
 *   dims == 1: every row of length n is rotated by n/2.
 *   dims == 2: every n x n image is rotated by (n/2, n/2).
 * ------------------------------------------------------------------------------------- */
int oracle_fftshift(const double* x, int64_t n, int64_t batch, int dims, double* out) {
    if (!x || !out || n < 2 || (n & 1) || batch < 1 || (dims != 1 && dims != 2)) return -1;
    if (x == out) return -1;
    const cplx* xi = (const cplx*)x;
    cplx* yo = (cplx*)out;
    int64_t h = n / 2;
    if (dims == 1) {
        for (int64_t b = 0; b < batch; ++b)
            for (int64_t k = 0; k < n; ++k) yo[b * n + (k + h) % n] = xi[b * n + k];
    } else {
        for (int64_t b = 0; b < batch; ++b)
            for (int64_t r = 0; r < n; ++r)
                for (int64_t c = 0; c < n; ++c)
                    yo[b * n * n + ((r + h) % n) * n + (c + h) % n] = xi[b * n * n + r * n + c];
    }
    return 0;
}

/* ---------------------------------------------------------------------------------------
 * General rotation, [Shift] "What is fftshift?" and its memory-move variants: every row
 * (ny == 1) or ny x nx image is rotated by (sy, sx), out[(y + sy) mod ny][(x + sx) mod nx] =
 * in[y][x], for any extents (odd ones included) and any shifts.  fftshift is the rotation by
 * (ny/2, nx/2) rounded down, ifftshift the rotation back.
 * ------------------------------------------------------------------------------------- */
int oracle_roll(const double* x, int64_t nx, int64_t ny, int64_t batch, int64_t sx, int64_t sy,
                double* out) {
    if (!x || !out || x == out || nx < 1 || ny < 1 || batch < 1) return -1;
    const cplx* xi = (const cplx*)x;
    cplx* yo = (cplx*)out;
    sx %= nx;
    if (sx < 0) sx += nx;
    sy %= ny;
    if (sy < 0) sy += ny;
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t y = 0; y < ny; ++y)
            for (int64_t c = 0; c < nx; ++c)
                yo[(b * ny + (y + sy) % ny) * nx + (c + sx) % nx] = xi[(b * ny + y) * nx + c];
    return 0;
}

/* Multiply by the chessboard (-1)^j (dims 1) or (-1)^(row+col) (dims 2), element-wise. */
int oracle_chessboard(const double* x, int64_t n, int64_t batch, int dims, double* out) {
    if (!x || !out || n < 1 || batch < 1 || (dims != 1 && dims != 2)) return -1;
    const cplx* xi = (const cplx*)x;
    cplx* yo = (cplx*)out;
    int64_t len = dims == 1 ? n : n * n;
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t i = 0; i < len; ++i) {
            int64_t parity = dims == 1 ? (i & 1) : (((i / n) + (i % n)) & 1);
            cplx v = xi[b * len + i];
            if (parity) {
                v.re = -v.re;
                v.im = -v.im;
            }
            yo[b * len + i] = v;
        }
    return 0;
}

/* ---------------------------------------------------------------------------------------
 * Band-limited real rows, [SHT] header comment and fftAnalysWGSL / fftSynthWGSL.
 *
 * Analysis (R2C): F_m = sum_{j<N} x_j exp(-2*pi*i*m*j/N), m = 0..mmax, computed as the
 *   forward complex FFT of the real row (imaginary part zero) truncated to m <= mmax.
 * Synthesis (C2R): assemble the Hermitian spectrum X_0 = Re F_0, X_m = F_m,
 *   X_{N-m} = conj F_m (1 <= m <= mmax), all other bins zero; x = Re(inverse FFT of X).
 *   Im F_0 is ignored, as the page reads only the real part of F_0.
 * Both take 0 <= mmax <= N/2.  The pages stop below N/2; at mmax = N/2 (even N) the Nyquist
 * bin is its own mirror (X_{N-N/2} = X_{N/2}), so Hermitian symmetry makes it real: the
 * synthesis uses Re F_{N/2} once (no conjugate partner) and ignores its imaginary part, as for
 * F_0.  Spectra here are row-major [batch][mmax+1].
 * ------------------------------------------------------------------------------------- */
int oracle_r2c(const double* xr, int64_t n, int64_t batch, int64_t mmax, double* F) {
    if (!xr || !F || !is_pow2(n) || n < 2 || batch < 1 || mmax < 0 || 2 * mmax > n) return -1;
    cplx* roots = make_roots(-1, n);
    if (!roots) return -1;
    int failed = 0;
#pragma omp parallel
    {
        cplx* in = (cplx*)malloc(sizeof(cplx) * (size_t)n);
        cplx* res = (cplx*)malloc(sizeof(cplx) * (size_t)n);
        if (!in || !res) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic)
            for (int64_t b = 0; b < batch; ++b) {
                for (int64_t j = 0; j < n; ++j) {
                    in[j].re = xr[b * n + j];
                    in[j].im = 0.0;
                }
                fft_rec(in, 1, n, roots, 1, res);
                memcpy((cplx*)F + b * (mmax + 1), res, sizeof(cplx) * (size_t)(mmax + 1));
            }
        }
        free(in);
        free(res);
    }
    free(roots);
    return failed ? -1 : 0;
}

int oracle_c2r(const double* F, int64_t n, int64_t batch, int64_t mmax, double* xr) {
    if (!F || !xr || !is_pow2(n) || n < 2 || batch < 1 || mmax < 0 || 2 * mmax > n) return -1;
    cplx* roots = make_roots(+1, n);
    if (!roots) return -1;
    int failed = 0;
#pragma omp parallel
    {
        cplx* spec = (cplx*)malloc(sizeof(cplx) * (size_t)n);
        cplx* res = (cplx*)malloc(sizeof(cplx) * (size_t)n);
        if (!spec || !res) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic)
            for (int64_t b = 0; b < batch; ++b) {
                const cplx* f = (const cplx*)F + b * (mmax + 1);
                memset(spec, 0, sizeof(cplx) * (size_t)n);
                spec[0].re = f[0].re; /* X_0 = Re F_0 */
                for (int64_t m = 1; m <= mmax; ++m) {
                    if (2 * m == n) {          /* Nyquist: real, its own mirror */
                        spec[m].re = f[m].re;
                        spec[m].im = 0.0;
                        continue;
                    }
                    spec[m] = f[m];            /* X_m = F_m */
                    spec[n - m].re = f[m].re;  /* X_{N-m} = conj F_m */
                    spec[n - m].im = -f[m].im;
                }
                fft_rec(spec, 1, n, roots, 1, res);
                for (int64_t j = 0; j < n; ++j) xr[b * n + j] = res[j].re;
            }
        }
        free(spec);
        free(res);
    }
    free(roots);
    return failed ? -1 : 0;
}

/* Direct band-limited sums, [SHT] dftAnalysWGSL / dftSynthWGSL:
 *   F_m = sum_j x_j exp(-2*pi*i*m*j/N)
 *   x_j = Re F_0 + 2 * sum_{m=1}^{mmax} Re(F_m exp(+2*pi*i*m*j/N)),
 * with the term of a Nyquist bin m = N/2 counted once, as Re F_{N/2} (-1)^j.
 * O(N * mmax) per row; any N >= 2 with 0 <= 2*mmax <= N. */
int oracle_r2c_direct(const double* xr, int64_t n, int64_t batch, int64_t mmax, double* F) {
    if (!xr || !F || n < 2 || batch < 1 || mmax < 0 || 2 * mmax > n) return -1;
#pragma omp parallel for schedule(dynamic)
    for (int64_t b = 0; b < batch; ++b) {
        for (int64_t m = 0; m <= mmax; ++m) {
            double sre = 0.0, sim = 0.0;
            for (int64_t j = 0; j < n; ++j) {
                cplx w = unit_root(-1, (int64_t)(((__int128)m * j) % n), n);
                sre += xr[b * n + j] * w.re;
                sim += xr[b * n + j] * w.im;
            }
            F[2 * (b * (mmax + 1) + m)] = sre;
            F[2 * (b * (mmax + 1) + m) + 1] = sim;
        }
    }
    return 0;
}

int oracle_c2r_direct(const double* F, int64_t n, int64_t batch, int64_t mmax, double* xr) {
    if (!F || !xr || n < 2 || batch < 1 || mmax < 0 || 2 * mmax > n) return -1;
#pragma omp parallel for schedule(dynamic)
    for (int64_t b = 0; b < batch; ++b) {
        const cplx* f = (const cplx*)F + b * (mmax + 1);
        for (int64_t j = 0; j < n; ++j) {
            double s = f[0].re;
            for (int64_t m = 1; m <= mmax; ++m) {
                if (2 * m == n) {  /* Nyquist: Re F_{N/2} (-1)^j, once */
                    s += (j & 1) ? -f[m].re : f[m].re;
                    continue;
                }
                cplx w = unit_root(+1, (int64_t)(((__int128)m * j) % n), n);
                s += 2.0 * (f[m].re * w.re - f[m].im * w.im);
            }
            xr[b * n + j] = s;
        }
    }
    return 0;
}
