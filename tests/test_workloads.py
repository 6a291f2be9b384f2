"""The seeded input generators: deterministic, right shapes/dtypes/distributions, and the
structured workloads carry their tones / plane waves where stated (checked with numpy's FFT)."""
import numpy as np

from fft_signal_processing_gb300 import workloads as wl


def test_deterministic_and_typed():
    a, b = wl.normal(3, 4, 64), wl.normal(3, 4, 64)
    np.testing.assert_array_equal(a, b)
    assert a.dtype == np.complex64 and a.shape == (4, 64)
    assert not np.array_equal(wl.normal(4, 4, 64), a)
    u = wl.uniform(1, 64, 1024)
    assert u.dtype == np.complex64 and -1 <= u.real.min() and u.real.max() < 1
    assert abs(u.real.mean()) < 0.02 and abs(u.imag.std() - 1 / np.sqrt(3)) < 0.01
    assert wl.real_normal(1, 3, 8).dtype == np.float32


def test_normal_moments():
    x = wl.normal(5, 256, 4096)
    assert abs(x.real.std() - 1) < 0.01 and abs(x.imag.mean()) < 0.01


def test_tones_have_three_spikes():
    n, batch = 1024, 6
    x = wl.tones(9, batch, n)
    f, phi = wl.tone_params(9, batch, n)
    X = np.abs(np.fft.fft(x.astype(np.complex128), axis=1))
    for r in range(batch):
        for k in set(f[r]):
            # unit tones exp(i(2 pi k j/n + phi)) -> n * |sum of exp(i phi)| at bin k
            amp = n * abs(np.sum(np.exp(1j * phi[r][f[r] == k])))
            assert abs(X[r, k] - amp) < 0.05 * n
        others = np.delete(X[r], f[r])
        # N(0, 0.1) per component -> |X_k| ~ 0.1 * sqrt(2n) (Rayleigh) away from the tones
        assert 0.5 < np.median(others) / (0.1 * np.sqrt(2 * n)) < 1.5


def test_spectrum_im_f0_is_zero():
    F = wl.spectrum(2, 16, 1365)
    assert F.shape == (16, 1366) and F.dtype == np.complex64
    assert np.all(F.imag[:, 0] == 0) and np.std(F.real) > 0.9


def test_image_plane_waves():
    n = 64
    img = wl.image(4, 2, n)
    ab, _ = wl.plane_wave_params(4, 2, n)
    X = np.abs(np.fft.fft2(img.astype(np.complex128)))
    for b in range(2):
        for a, bb in ab[b]:
            assert X[b, bb, a] > 0.5 * n * n  # row index = y frequency b, column = x frequency a
