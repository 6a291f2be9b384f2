"""fp64 CPU oracle for the batched FFT library (numpy front end over liboracle.so).

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference leg of ``bench.py`` may import this package.  The CUDA library and its Python
binding never import it, and it imports nothing from them.

Every function takes numpy arrays holding the exact values the GPU sees (complex64 / float32
are upcast to complex128 / float64, which is exact) and returns float64 / complex128 results.
Conventions (readings of the pages):

* ``fft``: X_k = sum_j x_j exp(s*2*pi*i*j*k/N), s = -1 forward, +1 inverse, unnormalised
  (Mota, "High Performance Fourier Transforms on GPUs with GLSL", §2.2 Eq. 5, without the
  1/N of the inverse; the WGSL fourier.ts Stockham kernels are unnormalised).
* ``fft_shifted``: forward with fftshift = rotation of every row (or image) by N/2
  ("The 1D fftshift in CUDA by chessboard multiplication", "What is fftshift?");
  inverse with shift = inverse transform, then multiply by the chessboard (-1)^j.
* ``r2c`` / ``c2r``: band-limited real analysis / synthesis of fourier.ts (header comment,
  fftAnalysWGSL / fftSynthWGSL), 0 <= 2*mmax <= N (mmax = N/2 adds the real Nyquist bin,
  counted once in the synthesis), spectra row-major [rows][mmax+1] or
  m-major [mmax+1][rows] (fourier.ts stores fm[m*NLAT + ilat]).
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        p = ctypes.c_void_p
        i64 = ctypes.c_int64
        ci = ctypes.c_int
        sig = {
            "oracle_dft": [p, i64, i64, ci, p],
            "oracle_dft_bins": [p, i64, ci, p, i64, p],
            "oracle_fft": [p, i64, i64, ci, p],
            "oracle_fft2d": [p, i64, i64, ci, p],
            "oracle_fft_any": [p, i64, i64, ci, p],
            "oracle_fftshift": [p, i64, i64, ci, p],
            "oracle_chessboard": [p, i64, i64, ci, p],
            "oracle_roll": [p, i64, i64, i64, i64, i64, p],
            "oracle_r2c": [p, i64, i64, i64, p],
            "oracle_c2r": [p, i64, i64, i64, p],
            "oracle_r2c_direct": [p, i64, i64, i64, p],
            "oracle_c2r_direct": [p, i64, i64, i64, p],
        }
        for name, args in sig.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = ci
        lib.oracle_num_threads.restype = ci
        lib.oracle_num_threads.argtypes = []
        lib.oracle_set_num_threads.restype = None
        lib.oracle_set_num_threads.argtypes = [ci]
        _LIB = lib
    return _LIB


def _c128(x):
    return np.ascontiguousarray(x, dtype=np.complex128)


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, name):
    if rc != 0:
        raise ValueError(f"oracle: {name} rejected its arguments")


def num_threads() -> int:
    """OpenMP threads the oracle uses."""
    return int(_lib().oracle_num_threads())


def set_num_threads(t: int) -> None:
    _lib().oracle_set_num_threads(int(t))


def dft(x, sign=-1):
    """Direct O(N^2) DFT of every row of x (last axis), any length N >= 1."""
    x = _c128(x)
    n = x.shape[-1]
    out = np.empty_like(x)
    _check(_lib().oracle_dft(_ptr(x), n, x.size // n, int(sign), _ptr(out)), "dft")
    return out


def dft_bins(row, bins, sign=-1):
    """Selected bins of one row, each by the direct O(N) sum."""
    row = _c128(row).ravel()
    bins = np.ascontiguousarray(bins, dtype=np.int64)
    out = np.empty(bins.shape, dtype=np.complex128)
    _check(_lib().oracle_dft_bins(_ptr(row), row.size, int(sign), _ptr(bins), bins.size,
                                  _ptr(out)), "dft_bins")
    return out


def fft(x, sign=-1):
    """Recursive radix-2 DIT FFT of every row of x (last axis, power-of-two length)."""
    x = _c128(x)
    n = x.shape[-1]
    out = np.empty_like(x)
    _check(_lib().oracle_fft(_ptr(x), n, x.size // n, int(sign), _ptr(out)), "fft")
    return out


def fft_any(x, sign=-1):
    """Mixed-radix recursive FFT of every row (last axis), any length N >= 1: radix = the
    smallest prime factor of N at each level, the direct sum for prime lengths."""
    x = _c128(x)
    n = x.shape[-1]
    out = np.empty_like(x)
    _check(_lib().oracle_fft_any(_ptr(x), n, x.size // n, int(sign), _ptr(out)), "fft_any")
    return out


def fft2d(x, sign=-1):
    """Row-column 2-D FFT of every n x n image (last two axes)."""
    x = _c128(x)
    n = x.shape[-1]
    if x.shape[-2] != n:
        raise ValueError("oracle.fft2d: images must be square")
    out = np.empty_like(x)
    _check(_lib().oracle_fft2d(_ptr(x), n, x.size // (n * n), int(sign), _ptr(out)), "fft2d")
    return out


def fft2d_rect(x, sign=-1):
    """Row-column 2-D FFT of every ny x nx image (last two axes, powers of two, rectangular
    allowed): the 1-D FFT of every row, then of every column (Mota §2.7 Eq. 19)."""
    x = _c128(x)
    rows = fft(x, sign)
    cols = fft(np.ascontiguousarray(np.swapaxes(rows, -1, -2)), sign)
    return np.ascontiguousarray(np.swapaxes(cols, -1, -2))


def fftshift(x, dims=1):
    """Rotate every row (dims=1) or image (dims=2) by n/2 (numpy-style fftshift, even n)."""
    x = _c128(x)
    n = x.shape[-1]
    out = np.empty_like(x)
    per = n if dims == 1 else n * n
    _check(_lib().oracle_fftshift(_ptr(x), n, x.size // per, int(dims), _ptr(out)),
           "fftshift")
    return out


def roll(x, shift_x, shift_y=0, dims=1):
    """Rotate every row (dims=1) or image (dims=2, last two axes ny x nx) by (shift_y, shift_x):
    out[(y + sy) mod ny][(x + sx) mod nx] = in[y][x]; any extents, odd ones included."""
    x = _c128(x)
    nx = x.shape[-1]
    ny = x.shape[-2] if dims == 2 else 1
    out = np.empty_like(x)
    _check(_lib().oracle_roll(_ptr(x), nx, ny, x.size // (nx * ny), int(shift_x), int(shift_y),
                              _ptr(out)), "roll")
    return out


def fftshift_any(x, dims=1, inverse=False):
    """fftshift (bin 0 to the middle: rotation by n/2 rounded down per axis) or, with
    inverse, ifftshift (the rotation back), of every row or ny x nx image."""
    sgn = -1 if inverse else 1
    nx = np.shape(x)[-1]
    ny = np.shape(x)[-2] if dims == 2 else 1
    return roll(x, sgn * (nx // 2), sgn * (ny // 2) if dims == 2 else 0, dims)


def chessboard(x, dims=1):
    """Multiply element-wise by (-1)^j (dims=1) or (-1)^(row+col) (dims=2)."""
    x = _c128(x)
    n = x.shape[-1]
    out = np.empty_like(x)
    per = n if dims == 1 else n * n
    _check(_lib().oracle_chessboard(_ptr(x), n, x.size // per, int(dims), _ptr(out)),
           "chessboard")
    return out


def transform(x, direction=-1, dims=1, shift=False):
    """What one exec of a C2C plan computes, in fp64.

    direction -1: forward; with shift, the output is fftshift(FFT(x)).
    direction +1: inverse; with shift, the output is IFFT(ifftshift(x)) (for even lengths the
    chessboard (-1)^j post-multiply of IFFT(x)).
    Rows whose length is not a power of two (dims 1) take the direct sum of Mota §2.2 Eq. 5.
    """
    n = np.shape(x)[-1]

    def t(v):
        if dims == 1:
            return fft(v, direction) if (n & (n - 1)) == 0 else dft(v, direction)
        return fft2d(v, direction) if np.shape(v)[-2] == n else fft2d_rect(v, direction)

    if not shift:
        return t(x)
    if direction == -1:
        return fftshift_any(t(x), dims)
    return t(fftshift_any(x, dims, inverse=True))


def to_mmajor(F):
    """Row-major spectrum [rows][mmax+1] -> m-major [mmax+1][rows] (fm[m*NLAT + ilat])."""
    return np.ascontiguousarray(np.asarray(F).T)


def from_mmajor(Fm):
    """m-major [mmax+1][rows] -> row-major [rows][mmax+1]."""
    return np.ascontiguousarray(np.asarray(Fm).T)


def r2c(x, mmax, layout="rowmajor"):
    """Band-limited analysis F_m, m = 0..mmax, of every real row (FFT path)."""
    x = _f64(x)
    n = x.shape[-1]
    rows = x.size // n
    F = np.empty((rows, mmax + 1), dtype=np.complex128)
    _check(_lib().oracle_r2c(_ptr(x), n, rows, int(mmax), _ptr(F)), "r2c")
    return to_mmajor(F) if layout == "mmajor" else F


def c2r(F, n, layout="rowmajor"):
    """Band-limited synthesis of real rows of length n from F_m (FFT path)."""
    F = _c128(from_mmajor(F) if layout == "mmajor" else F)
    rows, m1 = F.shape
    x = np.empty((rows, n), dtype=np.float64)
    _check(_lib().oracle_c2r(_ptr(F), n, rows, m1 - 1, _ptr(x)), "c2r")
    return x


def r2c_direct(x, mmax):
    """Direct band-limited analysis sum (row-major output)."""
    x = _f64(x)
    n = x.shape[-1]
    rows = x.size // n
    F = np.empty((rows, mmax + 1), dtype=np.complex128)
    _check(_lib().oracle_r2c_direct(_ptr(x), n, rows, int(mmax), _ptr(F)), "r2c_direct")
    return F


def c2r_direct(F, n):
    """Direct band-limited synthesis sum (row-major input)."""
    F = _c128(F)
    rows, m1 = F.shape
    x = np.empty((rows, n), dtype=np.float64)
    _check(_lib().oracle_c2r_direct(_ptr(F), n, rows, m1 - 1, _ptr(x)), "c2r_direct")
    return x


# ---- index maps (what the load and store epilogues do when no arithmetic intervenes) --------
def fourstep_order(x, n1):
    """The output order of the four-step decomposition n = n1*N2 + n2, k = k1 + N1*k2 (the
    CS598 page "Fast Fourier Transform on CPU and GPU", four-step remark): entry (k1, k2) of
    the [N1][N2] intermediate, held at k1*N2 + k2, is output bin k1 + N1*k2.  For every row."""
    x = np.asarray(x)
    n = x.shape[-1]
    n2 = n // n1
    return np.ascontiguousarray(
        np.swapaxes(x.reshape(x.shape[:-1] + (n1, n2)), -1, -2)).reshape(x.shape)


def hermitian_half(F, n):
    """The first n/2 bins X_0..X_{n/2-1} of the Hermitian spectrum a band-limited synthesis
    builds from F_0..F_mmax (fourier.ts header comment, fftSynthWGSL): X_0 = Re F_0, X_m = F_m
    for 1 <= m <= mmax, zero above (row-major F)."""
    F = _c128(F)
    rows, m1 = F.shape
    X = np.zeros((rows, n // 2), dtype=np.complex128)
    k = min(m1, n // 2)
    X[:, :k] = F[:, :k]
    X[:, 0] = X[:, 0].real
    return X


def pair_pack(x):
    """Two real rows per complex row (Mota, "High Performance Fourier Transforms on GPUs with
    GLSL", §2.6 Eq. 17): y = x_{2p} + i x_{2p+1}; an odd row count pairs the last row with
    zeros."""
    x = _f64(x)
    if x.shape[0] % 2:
        x = np.concatenate([x, np.zeros((1, x.shape[1]))])
    return x[0::2] + 1j * x[1::2]


def pair_unpack(Y, mmax, rows):
    """The two real rows' spectra from the transform of their packed row (the unpacking of
    Mota §2.6 Eq. 18, whose printed form is garbled; this is the form Hermitian symmetry
    gives): X1_k = (Y_k + conj Y_{n-k})/2, X2_k = (Y_k - conj Y_{n-k})/(2i), k = 0..mmax,
    as a row-major spectrum of `rows` rows."""
    Y = _c128(Y)
    n = Y.shape[-1]
    k = np.arange(mmax + 1)
    Yk, Yn = Y[:, k], np.conj(Y[:, (n - k) % n])
    F = np.empty((2 * Y.shape[0], mmax + 1), dtype=np.complex128)
    F[0::2] = (Yk + Yn) / 2
    F[1::2] = (Yk - Yn) / 2j
    return F[:rows]


def pair_assemble(F, n):
    """The packed spectrum Y_k = X1_k + i X2_k of two real rows, k = 0..n-1, each X the
    Hermitian extension of a band-limited F (X_0 = Re F_0, X_m = F_m and X_{n-m} = conj F_m
    for 1 <= m <= mmax, a Nyquist bin m = n/2 real, other bins zero; fourier.ts header
    comment).  The inverse transform of Y is x1 + i x2 (row-major F; odd row counts pair the
    last row with zeros)."""
    F = _c128(F)
    rows, m1 = F.shape
    if rows % 2:
        F = np.concatenate([F, np.zeros((1, m1), dtype=np.complex128)])
    X = np.zeros((F.shape[0], n), dtype=np.complex128)
    for m in range(m1):
        f = F[:, m].copy()
        if m == 0 or 2 * m == n:
            f = f.real.astype(np.complex128)
        X[:, m] = f
        if m != 0 and 2 * m != n:
            X[:, n - m] = np.conj(f)
    return X[0::2] + 1j * X[1::2]
