"""Seeded synthetic inputs for the transforms, on the host, as numpy arrays.

This module only draws random numbers and lays them out; it contains none of the transform
arithmetic, so the CUDA path and the fp64 oracle can both be fed from it without sharing any
of the method.  Every generator is deterministic in ``seed`` (numpy ``default_rng``).

The workloads follow the shapes and value distributions of the batched-FFT configurations
this library is measured on:

* ``uniform``  - re, im iid U[-1, 1)                     (1-D C2C, N = 1024 x 64 rows)
* ``normal``   - re, im iid N(0, 1)                      (1-D C2C, N = 4096 x 16384 rows)
* ``tones``    - per row 3 unit tones exp(i(2 pi f j/N + phi)), f integer U[0, N),
                 phi U[0, 2 pi), plus N(0, 0.1) noise per component (size sweep, batch*N = 2^26)
* ``spectrum`` - band-limited coefficients F_m, m = 0..mmax, re, im iid N(0, 1), Im F_0 = 0
                 (real-row synthesis / analysis, 2048 rows x 4096, mmax = 1365)
* ``image``    - N(0, 1) noise plus 4 unit plane waves exp(i(2 pi (a x + b y)/n + phi)),
                 (a, b) integer U[0, n)^2 (2-D C2C, 4096 x 4096)
* ``real_normal`` - real rows, iid N(0, 1) (input of a stand-alone analysis)
"""
import numpy as np

_CHUNK = 1 << 22  # points generated per chunk for the large workloads (bounds host memory)


def uniform(seed: int, batch: int, n: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    re = rng.uniform(-1.0, 1.0, size=(batch, n)).astype(np.float32)
    im = rng.uniform(-1.0, 1.0, size=(batch, n)).astype(np.float32)
    out = np.empty((batch, n), dtype=np.complex64)
    out.real, out.imag = re, im
    return out


def normal(seed: int, batch: int, n: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    out = np.empty((batch, n), dtype=np.complex64)
    rows_per = max(1, _CHUNK // max(n, 1))
    for r0 in range(0, batch, rows_per):
        r1 = min(batch, r0 + rows_per)
        out.real[r0:r1] = rng.standard_normal((r1 - r0, n), dtype=np.float32)
        out.imag[r0:r1] = rng.standard_normal((r1 - r0, n), dtype=np.float32)
    return out


def real_normal(seed: int, batch: int, n: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.standard_normal((batch, n), dtype=np.float32)


def tone_params(seed: int, batch: int, n: int, ntones: int = 3):
    """Integer frequencies f[batch, ntones] in [0, n) and phases phi in [0, 2 pi)."""
    rng = np.random.default_rng(seed)
    f = rng.integers(0, n, size=(batch, ntones), dtype=np.int64)
    phi = rng.uniform(0.0, 2.0 * np.pi, size=(batch, ntones))
    return f, phi


def tones(seed: int, batch: int, n: int, ntones: int = 3, noise: float = 0.1) -> np.ndarray:
    f, phi = tone_params(seed, batch, n, ntones)
    rng = np.random.default_rng(seed + 1_000_003)
    out = np.empty((batch, n), dtype=np.complex64)
    j = np.arange(n, dtype=np.int64)
    rows_per = max(1, _CHUNK // max(n, 1))
    for r0 in range(0, batch, rows_per):
        r1 = min(batch, r0 + rows_per)
        acc = np.zeros((r1 - r0, n), dtype=np.complex128)
        for t in range(ntones):
            # phase 2 pi (f j mod n)/n + phi, reduced in integers before the float multiply
            q = (f[r0:r1, t, None] * j[None, :]) % n
            acc += np.exp(1j * (2.0 * np.pi * q / n + phi[r0:r1, t, None]))
        acc.real += noise * rng.standard_normal((r1 - r0, n))
        acc.imag += noise * rng.standard_normal((r1 - r0, n))
        out[r0:r1] = acc.astype(np.complex64)
    return out


def spectrum(seed: int, rows: int, mmax: int) -> np.ndarray:
    """Row-major coefficients [rows][mmax+1] (complex64), Im F_0 = 0."""
    rng = np.random.default_rng(seed)
    F = np.empty((rows, mmax + 1), dtype=np.complex64)
    F.real = rng.standard_normal((rows, mmax + 1), dtype=np.float32)
    F.imag = rng.standard_normal((rows, mmax + 1), dtype=np.float32)
    F.imag[:, 0] = 0.0
    return F


def plane_wave_params(seed: int, batch: int, n: int, nwaves: int = 4):
    rng = np.random.default_rng(seed)
    ab = rng.integers(0, n, size=(batch, nwaves, 2), dtype=np.int64)
    phi = rng.uniform(0.0, 2.0 * np.pi, size=(batch, nwaves))
    return ab, phi


def image(seed: int, batch: int, n: int, nwaves: int = 4) -> np.ndarray:
    """Images [batch][n][n] (complex64): row index y, column index x."""
    ab, phi = plane_wave_params(seed, batch, n, nwaves)
    rng = np.random.default_rng(seed + 1_000_003)
    out = np.empty((batch, n, n), dtype=np.complex64)
    x = np.arange(n, dtype=np.int64)
    rows_per = max(1, _CHUNK // n)
    for b in range(batch):
        for y0 in range(0, n, rows_per):
            y1 = min(n, y0 + rows_per)
            y = np.arange(y0, y1, dtype=np.int64)
            acc = rng.standard_normal((y1 - y0, n)) + 1j * rng.standard_normal((y1 - y0, n))
            for w in range(nwaves):
                a, bb = ab[b, w]
                q = (a * x[None, :] + bb * y[:, None]) % n
                acc += np.exp(1j * (2.0 * np.pi * q / n + phi[b, w]))
            out[b, y0:y1] = acc.astype(np.complex64)
    return out
