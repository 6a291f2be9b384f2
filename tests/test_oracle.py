"""Pins for the fp64 oracle, against facts the pages and the mathematics fix (CPU only).

Each check is independent of the oracle's own code: a printed worked example, the closed
4-point form, brute force on tiny sizes, numpy's FFT (a library routine), closed forms
(delta, tone, plane wave, single real mode) and invariants (linearity, Parseval, round trip,
chessboard = rotation, Hermitian symmetry).
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def crand(*shape):
    return RNG.standard_normal(shape) + 1j * RNG.standard_normal(shape)


def rel(a, b):
    return np.linalg.norm(np.ravel(a - b)) / max(np.linalg.norm(np.ravel(b)), 1e-300)


# --- Mota §2.2 worked example -----------------------------------------------------------------
def _load_golden(name):
    x, X = {}, {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            tag, i, re, im = line.split()
            (x if tag == "x" else X)[int(i)] = complex(float(re), float(im))
    n = len(x)
    return (np.array([x[i] for i in range(n)]), np.array([X[i] for i in range(n)]))


def test_worked_example_n8():
    x, X = _load_golden("dft_worked_example_n8.txt")
    for f in (oracle.fft, oracle.dft):
        np.testing.assert_allclose(f(x[None], -1)[0], X, atol=1e-3)
    # with the exact samples cos(2 pi n/8) the printed answer holds to rounding
    xe = np.cos(2 * np.pi * np.arange(8) / 8)
    np.testing.assert_allclose(oracle.fft(xe[None], -1)[0], X, atol=1e-12)


# --- Mota §2.3 Eq. 7: the 4-point DFT written out -------------------------------------------
@pytest.mark.parametrize("sign", [-1, 1])
def test_four_point_closed_form(sign):
    x = crand(16, 4)
    x0, x1, x2, x3 = x.T
    i = 1j * (-sign)  # Eq. 7 is the forward transform; the inverse flips i
    X = np.stack([x0 + x1 + x2 + x3,
                  x0 - i * x1 - x2 + i * x3,
                  x0 - x1 + x2 - x3,
                  x0 + i * x1 - x2 - i * x3], axis=1)
    np.testing.assert_allclose(oracle.fft(x, sign), X, atol=1e-13)
    np.testing.assert_allclose(oracle.dft(x, sign), X, atol=1e-13)


# --- brute force and a library FFT ----------------------------------------------------------
@pytest.mark.parametrize("n", [1, 2, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("sign", [-1, 1])
def test_fft_matches_direct_dft(n, sign):
    x = crand(3, n)
    # an independent direct sum written in numpy (outer product of indices)
    j = np.arange(n)
    W = np.exp(sign * 2j * np.pi * np.outer(j, j) / n)
    ref = x @ W
    assert rel(oracle.dft(x, sign), ref) < 1e-13
    assert rel(oracle.fft(x, sign), ref) < 1e-13


@pytest.mark.parametrize("n", [3, 5, 6, 12])
def test_dft_non_power_of_two_vs_numpy(n):
    x = crand(2, n)
    assert rel(oracle.dft(x, -1), np.fft.fft(x)) < 1e-13


@pytest.mark.parametrize("logn", list(range(1, 17)) + [20])
def test_fft_matches_numpy(logn):
    n = 1 << logn
    rows = max(1, (1 << 16) // n)
    x = crand(rows, n)
    assert rel(oracle.fft(x, -1), np.fft.fft(x)) < 1e-14
    assert rel(oracle.fft(x, +1), np.fft.ifft(x) * n) < 1e-14


def test_fft_rejects_non_power_of_two():
    with pytest.raises(ValueError):
        oracle.fft(crand(1, 6))


# --- closed forms -----------------------------------------------------------------------------
@pytest.mark.parametrize("n", [2, 16, 1024, 1 << 15])
def test_delta(n):
    x = np.zeros((1, n), complex)
    x[0, 0] = 1
    np.testing.assert_array_equal(oracle.fft(x, -1), np.ones((1, n)))
    j0 = 3 % n
    x = np.zeros((1, n), complex)
    x[0, j0] = 1
    k = np.arange(n)
    np.testing.assert_allclose(oracle.fft(x, -1)[0], np.exp(-2j * np.pi * j0 * k / n),
                               atol=1e-12)


@pytest.mark.parametrize("n", [8, 256, 4096])
@pytest.mark.parametrize("sign", [-1, 1])
def test_tone_gives_delta(n, sign):
    k0 = (5 * n) // 7
    j = np.arange(n)
    x = np.exp(-sign * 2j * np.pi * k0 * j / n)[None]
    X = oracle.fft(x, sign)[0]
    ref = np.zeros(n, complex)
    ref[k0] = n
    assert np.max(np.abs(X - ref)) < 1e-9 * n


def test_linearity():
    x, y = crand(4, 512), crand(4, 512)
    a, b = 0.3 - 1.2j, -2.0 + 0.5j
    assert rel(oracle.fft(a * x + b * y), a * oracle.fft(x) + b * oracle.fft(y)) < 1e-14


@pytest.mark.parametrize("n", [64, 8192])
def test_parseval(n):
    x = crand(2, n)
    X = oracle.fft(x)
    np.testing.assert_allclose(np.sum(np.abs(X) ** 2, axis=1),
                               n * np.sum(np.abs(x) ** 2, axis=1), rtol=1e-12)


@pytest.mark.parametrize("n", [2, 128, 1 << 14])
def test_round_trip_is_n_times_identity(n):
    x = crand(3, n)
    assert rel(oracle.fft(oracle.fft(x, -1), +1), n * x) < 1e-14


def test_dft_bins_match_fft():
    n = 1 << 12
    x = crand(1, n)
    bins = np.array([0, 1, 7, n // 2, n - 1, 1234])
    np.testing.assert_allclose(oracle.dft_bins(x[0], bins, -1), oracle.fft(x, -1)[0, bins],
                               atol=1e-9)


# --- chessboard fftshift ("The 1D fftshift in CUDA by chessboard multiplication") -----------
@pytest.mark.parametrize("n", [2, 8, 4096])
def test_fftshift_matches_numpy(n):
    x = crand(3, n)
    np.testing.assert_array_equal(oracle.fftshift(x, 1), np.fft.fftshift(x, axes=-1))
    img = crand(2, 8, 8)
    np.testing.assert_array_equal(oracle.fftshift(img, 2), np.fft.fftshift(img, axes=(-2, -1)))


@pytest.mark.parametrize("n", [2, 16, 4096])
def test_chessboard_premultiply_equals_shift(n):
    x = crand(4, n)
    lhs = oracle.fft(oracle.chessboard(x, 1), -1)
    rhs = oracle.fftshift(oracle.fft(x, -1), 1)
    assert rel(lhs, rhs) < 1e-14
    # inverse with shift undoes forward with shift up to the factor N
    y = oracle.transform(oracle.transform(x, -1, 1, True), +1, 1, True)
    assert rel(y, n * x) < 1e-14


@pytest.mark.parametrize("n", [6, 12, 1000])
def test_any_length_transform_and_shift(n):
    """Lengths that are not powers of two: the direct sum against a brute-force outer product
    written here (small n) or numpy's FFT; the chessboard identity still holds for even n."""
    x = crand(3, n)
    if n <= 64:
        j = np.arange(n)
        ref = x @ np.exp(-2j * np.pi * np.outer(j, j) / n)
    else:
        ref = np.fft.fft(x)
    assert rel(oracle.transform(x, -1), ref) < 1e-12
    assert rel(oracle.transform(x, +1), np.fft.ifft(x) * n) < 1e-12
    lhs = oracle.dft(oracle.chessboard(x, 1), -1)
    assert rel(lhs, oracle.transform(x, -1, 1, True)) < 1e-12
    assert rel(lhs, np.fft.fftshift(ref, axes=-1)) < 1e-12
    y = oracle.transform(oracle.transform(x, -1, 1, True), +1, 1, True)
    assert rel(y, n * x) < 1e-12


@pytest.mark.parametrize("n,mmax", [(7, 3), (12, 5), (1000, 499), (999, 100)])
def test_direct_band_limited_sums_any_length(n, mmax):
    """Real rows of any length: the direct analysis/synthesis sums against numpy's real FFT
    (rfft truncated to mmax; irfft of the zero-padded spectrum times n, which also ignores
    Im F_0, as fourier.ts's synthesis does)."""
    rng = np.random.default_rng(n)
    x = rng.standard_normal((3, n))
    F = oracle.r2c_direct(x, mmax)
    assert rel(F, np.fft.rfft(x)[:, :mmax + 1]) < 1e-12
    G = rng.standard_normal((3, mmax + 1)) + 1j * rng.standard_normal((3, mmax + 1))
    pad = np.zeros((3, n // 2 + 1), complex)
    pad[:, :mmax + 1] = G
    pad[:, 0] = G[:, 0].real
    assert rel(oracle.c2r_direct(G, n), np.fft.irfft(pad, n) * n) < 1e-12


@pytest.mark.parametrize("shape", [(3, 7), (2, 8), (2, 5, 6), (1, 9, 4), (2, 8, 8)])
def test_roll_fftshift_ifftshift_match_numpy(shape):
    """The general rotation against numpy's fftshift / ifftshift (library routines): odd and
    even extents, rows and rectangular images."""
    x = crand(*shape)
    dims = 2 if len(shape) == 3 else 1
    axes = (-2, -1) if dims == 2 else (-1,)
    np.testing.assert_array_equal(oracle.fftshift_any(x, dims), np.fft.fftshift(x, axes=axes))
    np.testing.assert_array_equal(oracle.fftshift_any(x, dims, inverse=True),
                                  np.fft.ifftshift(x, axes=axes))
    np.testing.assert_array_equal(oracle.roll(x, 2, 1 if dims == 2 else 0, dims),
                                  np.roll(x, (1, 2) if dims == 2 else 2, axis=axes))


@pytest.mark.parametrize("n", [7, 9, 1001])
def test_odd_length_shift_by_complex_exponential(n):
    """For odd n the shifted transform is the transform of x_j * exp(+2*pi*i*j*(n//2)/n)
    (forward), and IFFT(ifftshift(X)) is IFFT(X)_j * exp(-2*pi*i*j*(n//2)/n) (inverse)."""
    x = crand(2, n)
    e = np.exp(2j * np.pi * np.arange(n) * (n // 2) / n)
    assert rel(oracle.transform(x, -1, 1, True), oracle.dft(x * e, -1)) < 1e-12
    assert rel(oracle.transform(x, +1, 1, True), oracle.dft(x, +1) / e) < 1e-12
    assert rel(oracle.transform(oracle.transform(x, -1, 1, True), +1, 1, True), n * x) < 1e-12


@pytest.mark.parametrize("n", [8, 12, 1024])
def test_nyquist_bin_full_half_spectrum(n):
    """mmax = n/2: the full n/2 + 1 half spectrum against numpy's rfft / irfft (library
    routines; irfft also drops the imaginary parts of bins 0 and n/2), both oracle paths."""
    rng = np.random.default_rng(n)
    x = rng.standard_normal((3, n))
    h = n // 2
    assert rel(oracle.r2c_direct(x, h), np.fft.rfft(x)) < 1e-12
    if n & (n - 1) == 0:
        assert rel(oracle.r2c(x, h), np.fft.rfft(x)) < 1e-12
    G = rng.standard_normal((3, h + 1)) + 1j * rng.standard_normal((3, h + 1))
    ref = np.fft.irfft(G, n) * n
    assert rel(oracle.c2r_direct(G, n), ref) < 1e-12
    if n & (n - 1) == 0:
        assert rel(oracle.c2r(G, n), ref) < 1e-12
    # a lone Nyquist coefficient synthesises Re F_{n/2} (-1)^j
    N = np.zeros((1, h + 1), complex)
    N[0, h] = 2.5 - 7j
    np.testing.assert_allclose(oracle.c2r_direct(N, n)[0], 2.5 * (-1.0) ** np.arange(n))


@pytest.mark.parametrize("ny,nx", [(2, 8), (16, 4), (64, 32)])
def test_rectangular_2d_matches_numpy_and_separability(ny, nx):
    x = crand(2, ny, nx)
    assert rel(oracle.fft2d_rect(x, -1), np.fft.fft2(x)) < 1e-13
    assert rel(oracle.fft2d_rect(x, +1), np.fft.ifft2(x) * nx * ny) < 1e-13
    u, v = crand(1, ny)[0], crand(1, nx)[0]
    sep = oracle.fft2d_rect(np.outer(u, v)[None], -1)[0]
    assert rel(sep, np.outer(oracle.fft(u[None])[0], oracle.fft(v[None])[0])) < 1e-13
    # the shifted transform: 2-D fftshift of the transform; the inverse undoes it up to nx*ny
    y = oracle.transform(x, -1, 2, True)
    assert rel(y, np.fft.fftshift(np.fft.fft2(x), axes=(-2, -1))) < 1e-13
    assert rel(oracle.transform(y, +1, 2, True), nx * ny * x) < 1e-13


@pytest.mark.parametrize("n", [1, 2, 3, 6, 7, 12, 30, 97, 100, 210, 1000, 1024, 3 * 5 * 7 * 11,
                               2 * 8191, 60000, 100000, 3 ** 12, 10 ** 6, (1 << 20) - 1])
@pytest.mark.parametrize("sign", [-1, 1])
def test_mixed_radix_fft_any_length(n, sign):
    """The mixed-radix FFT against numpy's FFT (a library routine) at composite, prime and
    power-of-two lengths, against the direct sum at small lengths and against the radix-2
    recursion at powers of two."""
    x = crand(2, n)
    ref = np.fft.fft(x) if sign < 0 else np.fft.ifft(x) * n
    got = oracle.fft_any(x, sign)
    assert rel(got, ref) < 1e-12
    if n <= 210:
        assert rel(got, oracle.dft(x, sign)) < 1e-12
    if n & (n - 1) == 0:
        assert rel(got, oracle.fft(x, sign)) < 1e-13


def test_chessboard_values():
    x = np.ones((1, 6), complex)
    np.testing.assert_array_equal(oracle.chessboard(x, 1)[0], [1, -1, 1, -1, 1, -1])
    img = np.ones((1, 2, 2), complex)
    np.testing.assert_array_equal(oracle.chessboard(img, 2)[0], [[1, -1], [-1, 1]])


def test_shifted_tone_lands_at_k_plus_half():
    n, k0 = 64, 5
    x = np.exp(2j * np.pi * k0 * np.arange(n) / n)[None]
    X = oracle.transform(x, -1, 1, True)[0]
    assert np.argmax(np.abs(X)) == (k0 + n // 2) % n


# --- 2-D (Mota §2.7 Eq. 19) -------------------------------------------------------------------
def test_fft2d_matches_numpy_and_separability():
    n = 32
    img = crand(2, n, n)
    assert rel(oracle.fft2d(img, -1), np.fft.fft2(img)) < 1e-14
    assert rel(oracle.fft2d(img, +1), np.fft.ifft2(img) * n * n) < 1e-14
    u, v = crand(n), crand(n)
    lhs = oracle.fft2d(np.outer(u, v)[None], -1)[0]
    rhs = np.outer(oracle.fft(u[None])[0], oracle.fft(v[None])[0])
    assert rel(lhs, rhs) < 1e-14


def test_plane_wave_and_2d_shift():
    n, a, b = 16, 3, 11
    y, x = np.meshgrid(np.arange(n), np.arange(n), indexing="ij")
    img = np.exp(2j * np.pi * (a * x + b * y) / n)[None]
    X = oracle.fft2d(img, -1)[0]
    ref = np.zeros((n, n), complex)
    ref[b, a] = n * n
    assert np.max(np.abs(X - ref)) < 1e-10
    Xs = oracle.transform(img, -1, 2, True)[0]
    assert np.unravel_index(np.argmax(np.abs(Xs)), Xs.shape) == ((b + n // 2) % n,
                                                                  (a + n // 2) % n)
    assert rel(oracle.fft2d(oracle.chessboard(img, 2), -1), oracle.fftshift(X[None], 2)) < 1e-14
    rt = oracle.transform(oracle.transform(img, -1, 2, True), +1, 2, True)
    assert rel(rt, n * n * img) < 1e-14


# --- band-limited real rows (fourier.ts) ------------------------------------------------------
@pytest.mark.parametrize("n,mmax", [(2, 0), (8, 3), (64, 20), (4096, 1365)])
def test_r2c_is_truncated_c2c_and_direct_sum(n, mmax):
    x = RNG.standard_normal((3, n))
    F = oracle.r2c(x, mmax)
    assert rel(F, np.fft.fft(x)[:, :mmax + 1]) < 1e-14
    if n <= 64:
        assert rel(F, oracle.r2c_direct(x, mmax)) < 1e-13


def test_real_row_spectrum_is_hermitian():
    n = 256
    X = oracle.fft(RNG.standard_normal((2, n)).astype(complex))
    np.testing.assert_allclose(X[:, 1:], np.conj(X[:, :0:-1]), atol=1e-12)


@pytest.mark.parametrize("n,mmax", [(2, 0), (8, 3), (64, 31), (256, 85)])
def test_c2r_matches_direct_sum(n, mmax):
    F = crand(3, mmax + 1)
    assert rel(oracle.c2r(F, n), oracle.c2r_direct(F, n)) < 1e-13


def test_c2r_single_mode_is_a_cosine():
    n, m, A, th = 128, 9, 0.75, 0.4
    F = np.zeros((1, 20), complex)
    F[0, m] = A * np.exp(1j * th)
    j = np.arange(n)
    np.testing.assert_allclose(oracle.c2r(F, n)[0], 2 * A * np.cos(2 * np.pi * m * j / n + th),
                               atol=1e-12)
    F = np.zeros((1, 20), complex)
    F[0, 0] = 1.5 + 7.0j  # only Re F_0 is used
    np.testing.assert_allclose(oracle.c2r(F, n)[0], np.full(n, 1.5), atol=1e-13)


def test_analysis_of_synthesis():
    n, mmax = 512, 170
    F = crand(4, mmax + 1)
    G = oracle.r2c(oracle.c2r(F, n), mmax)
    np.testing.assert_allclose(G[:, 1:], n * F[:, 1:], rtol=1e-12, atol=1e-9)
    np.testing.assert_allclose(G[:, 0], n * F[:, 0].real, atol=1e-9)


def test_mmajor_layout_is_fm_m_times_nlat_plus_ilat():
    nlat, mmax = 5, 3
    F = crand(nlat, mmax + 1)
    flat = oracle.to_mmajor(F).ravel()
    for ilat in range(nlat):
        for m in range(mmax + 1):
            assert flat[m * nlat + ilat] == F[ilat, m]
    np.testing.assert_array_equal(oracle.from_mmajor(oracle.to_mmajor(F)), F)
    x = RNG.standard_normal((nlat, 16))
    np.testing.assert_array_equal(oracle.r2c(x, 5, "mmajor"), oracle.to_mmajor(oracle.r2c(x, 5)))


@pytest.mark.parametrize("bad", [(8, 5), (8, -1), (6, 1)])
def test_band_limit_rejected(bad):
    n, mmax = bad
    with pytest.raises(ValueError):
        oracle.r2c(np.zeros((1, n)), mmax)


# ---- index maps used by the bit-exact epilogue tests ------------------------------------------
def test_fourstep_order_is_the_four_step_output_map():
    """The four-step FFT written out with numpy's FFT (columns, twiddle w_n^{n2*k1}, rows) gives
    the DFT only when its [N1][N2] result is read through fourstep_order."""
    rng = np.random.default_rng(40)
    n1, n2 = 8, 16
    n = n1 * n2
    x = rng.standard_normal((3, n)) + 1j * rng.standard_normal((3, n))
    a = x.reshape(3, n1, n2)
    y = np.fft.fft(a, axis=1)                                  # over n1, for each n2
    y *= np.exp(-2j * np.pi * np.outer(np.arange(n1), np.arange(n2)) / n)  # w_n^{k1*n2}
    z = np.fft.fft(y, axis=2).reshape(3, n)                    # over n2: [k1][k2]
    np.testing.assert_allclose(oracle.fourstep_order(z, n1), oracle.fft(x), atol=1e-9)
    assert oracle.fourstep_order(np.arange(8.0)[None], 2).tolist() == [[0, 4, 1, 5, 2, 6, 3, 7]]


def test_pair_pack_unpack_gives_both_rows_spectra():
    rng = np.random.default_rng(41)
    for rows, n, mmax in ((5, 64, 32), (4, 60, 20), (1, 16, 3)):
        x = rng.standard_normal((rows, n))
        Y = oracle.fft_any(oracle.pair_pack(x), -1)
        np.testing.assert_allclose(oracle.pair_unpack(Y, mmax, rows),
                                   np.fft.fft(x)[:, :mmax + 1], atol=1e-9)


def test_pair_assemble_synthesises_both_rows():
    rng = np.random.default_rng(42)
    for rows, n, mmax in ((5, 64, 32), (4, 60, 30), (3, 64, 10)):
        F = rng.standard_normal((rows, mmax + 1)) + 1j * rng.standard_normal((rows, mmax + 1))
        y = oracle.fft_any(oracle.pair_assemble(F, n), +1)
        x = np.empty((2 * y.shape[0], n))
        x[0::2], x[1::2] = y.real, y.imag
        np.testing.assert_allclose(x[:rows], oracle.c2r_direct(F, n), atol=1e-9)


def test_hermitian_half_is_the_lower_half_of_the_synthesis_spectrum():
    rng = np.random.default_rng(43)
    n, mmax = 32, 12
    F = rng.standard_normal((3, mmax + 1)) + 1j * rng.standard_normal((3, mmax + 1))
    Y = oracle.pair_assemble(F[:1], n)  # a row paired with zeros: Y = X of that row
    np.testing.assert_array_equal(oracle.hermitian_half(F, n)[:1], Y[:, :n // 2])
    assert oracle.hermitian_half(F, n)[0, 0].imag == 0
    assert np.all(oracle.hermitian_half(F[:, :3], n)[:, 3:] == 0)
