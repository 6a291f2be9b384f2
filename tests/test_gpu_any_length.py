"""GPU parity of rows whose length is not a power of two (the mixed-radix and chirp-z paths)
against the fp64 oracle's direct sums, through the C ABI: complex rows against the DFT of Mota,
"High Performance Fourier Transforms on GPUs with GLSL", §2.2 Eq. 5; band-limited real rows
against the direct analysis/synthesis sums of fourier.ts (dftAnalysWGSL / dftSynthWGSL), both
spectrum layouts.

Lengths span every chirp-z size m = 8 .. 16384 (m the power of two >= 2n - 1), including
n just above and below powers of two, odd and even n, ragged batches, both directions, the
chessboard shift (even n), in place, and one full benchmark-sized batch with sampled rows.
Lengths whose prime factors are 2, 3, 5 and 7 (up to 8192) run both on their default
mixed-radix path and, forced with GBFFT_FORCE_PATH=chirpz, on the chirp-z path.
"""
import os

import numpy as np
import pytest

import oracle
from parity import assert_parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__

    __graft_entry__.build()


def fx():
    import fft_signal_processing_gb300 as m

    return m


def wl():
    from fft_signal_processing_gb300 import workloads

    return workloads


def smooth(n):
    for f in (2, 3, 5, 7):
        while n % f == 0:
            n //= f
    return n == 1


def mixed_split_exists(n):
    """The planner's four-step split of a long smooth length: a divisor N1 <= min(512, sqrt n)
    with n / N1 <= 8192."""
    return any(n % d == 0 and n // d <= 8192 for d in range(2, min(512, int(n ** 0.5)) + 1))


def expected_path(n, real=False):
    """The path prefix the planner must choose: mixed-radix (one pass up to 8192 points, the
    four-step above) for lengths whose prime factors are 2, 3, 5, 7, chirp-z otherwise or when
    forced; the same for complex and real rows."""
    if os.environ.get("GBFFT_FORCE_PATH") == "chirpz" or not smooth(n):
        return "path=bluestein"
    if n <= 8192 or (n <= 1 << 20 and mixed_split_exists(n)):
        return "path=mixed"
    return "path=bluestein"


@pytest.fixture(params=["default", "chirpz"])
def route(request, monkeypatch):
    """The default path choice, and the chirp-z path forced (GBFFT_FORCE_PATH=chirpz); lengths
    with a prime factor above 7 take the chirp-z path either way and run once."""
    if request.param == "chirpz":
        monkeypatch.setenv("GBFFT_FORCE_PATH", "chirpz")
    return request.param


def skip_same(n, route):
    if route == "chirpz" and not smooth(n):
        pytest.skip("the default path of this length is the chirp-z path")


def gpu_c2c(x, n, batch, direction, shift=False, inplace=False):
    m = fx()
    p = m.Plan(n, batch, 1, direction, shift=shift)
    assert expected_path(n) in p.describe()
    xd = torch.from_numpy(np.ascontiguousarray(x, dtype=np.complex64)).cuda()
    if inplace:
        p.c2c(xd, out=xd)
        y = xd
    else:
        y = p.c2c(xd)
    torch.cuda.synchronize()
    p.check()
    return y.cpu().numpy()


LENGTHS = [3, 5, 6, 7, 12, 31, 33, 100, 127, 129, 255, 257, 1000, 1023, 1025, 2047, 3000,
           4095, 4097, 6000, 8191]


@pytest.mark.parametrize("n", LENGTHS)
@pytest.mark.parametrize("direction", [-1, 1])
def test_any_length_grid(n, direction, route):
    skip_same(n, route)
    batch = 37 if n <= 1100 else 3  # ragged against every rows-per-CTA count
    x = wl().normal(7000 + n, batch, n)
    got = gpu_c2c(x, n, batch, direction)
    assert_parity(got, oracle.transform(x, direction), n, f"n={n} dir={direction}")


@pytest.mark.parametrize("n", [3, 6, 7, 100, 1000, 1001, 4098, 4099, 8190, 8191, 3 * 5 * 7 * 9])
@pytest.mark.parametrize("direction", [-1, 1])
def test_any_length_shift_in_place(n, direction, route):
    """Even lengths: the chessboard; odd lengths: the complex exponentials (folded into the
    chirp tables, or the phase table of the mixed-radix path); against fftshift(DFT(x)) and
    IFFT(ifftshift(X)) of the oracle."""
    skip_same(n, route)
    batch = 5
    x = wl().uniform(7100 + n, batch, n)
    got = gpu_c2c(x, n, batch, direction, shift=True, inplace=True)
    assert_parity(got, oracle.transform(x, direction, 1, True), n, f"shift n={n}")
    if direction == -1:  # bin 0 lands at index n//2
        y = gpu_c2c(np.ones((1, n), np.complex64), n, 1, -1, shift=True)
        assert np.argmax(np.abs(y[0])) == n // 2


@pytest.mark.parametrize("n", [3, 1000, 8191, 7168])
def test_any_length_round_trip_and_tones(n, route):
    skip_same(n, route)
    batch = 4
    x = wl().tones(7200 + n, batch, n)
    y = gpu_c2c(x, n, batch, -1)
    z = gpu_c2c(y, n, batch, +1)
    assert_parity(z, n * x.astype(np.complex128), n, f"round trip n={n}")
    f, phi = wl().tone_params(7200 + n, batch, n)
    for r in range(batch):  # unit tones land on their bins with magnitude ~ n
        for k in set(f[r]):
            amp = n * abs(np.sum(np.exp(1j * phi[r][f[r] == k])))
            assert abs(abs(y[r, k]) - amp) < 0.05 * n + 0.6 * (2 * n) ** 0.5


def test_any_length_full_batch_sampled():
    """The benchmark's any-length workload at full size (n = 1000, batch = 2^26 // 1000),
    sampled rows against the oracle's direct sum."""
    m = fx()
    n = 1000
    batch = (1 << 26) // n
    x = wl().tones(7300, batch, n)
    p = m.Plan(n, batch, 1, m.FORWARD)
    y = p.c2c(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    p.check()
    rng = np.random.default_rng(7300)
    rows = np.array(sorted({0, batch - 1, batch // 2, *rng.integers(0, batch, 29).tolist()}))
    ys = y[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert_parity(ys, oracle.transform(x[rows], -1), n, "n=1000 full batch")


@pytest.mark.parametrize("n", [12, 100, 1000])
@pytest.mark.parametrize("direction,shift", [(-1, False), (1, True)])
def test_mixed_small_shape_large_batches(n, direction, shift):
    """Batches of at least 8192 rows of at most 1024 points take the mixed-radix kernel's
    128-thread shape: ragged against its rows per CTA, sampled rows against the oracle."""
    m = fx()
    batch = 8192 + 37
    p = m.Plan(n, batch, 1, direction, shift=shift)
    assert "path=mixed" in p.describe() and "threads=128" in p.describe()
    x = wl().normal(7320 + n, batch, n)
    y = p.c2c(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    p.check()
    rng = np.random.default_rng(n)
    rows = np.array(sorted({0, batch - 1, *rng.integers(0, batch, 30).tolist()}))
    ys = y[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert_parity(ys, oracle.transform(x[rows], direction, 1, shift), n, f"small shape n={n}")


@pytest.mark.parametrize("pairing", [False, True])
def test_mixed_small_shape_real_rows(pairing):
    """Real rows of 100 points, 16384 + 5 of them (at least 8192 transforms either way):
    synthesis then analysis on the 128-thread shape, sampled rows against the direct sums."""
    m = fx()
    n, rows, mmax = 100, 16389, 50
    syn = m.Plan(n, rows, 1, m.INVERSE, layout=m.LAYOUT_REAL_MMAJOR, mmax=mmax, pairing=pairing)
    ana = m.Plan(n, rows, 1, m.FORWARD, layout=m.LAYOUT_REAL_ROWMAJOR, mmax=mmax, pairing=pairing)
    assert "threads=128" in syn.describe() and "threads=128" in ana.describe()
    F = wl().spectrum(7330, rows, mmax)
    x = syn.c2r(torch.from_numpy(np.ascontiguousarray(oracle.to_mmajor(F), dtype=np.complex64)).cuda())
    G = ana.r2c(x)
    torch.cuda.synchronize()
    syn.check()
    ana.check()
    pick = np.array(sorted({0, rows - 1, *np.random.default_rng(7330).integers(0, rows, 30).tolist()}))
    xs = x.cpu().numpy()
    ref_x = oracle.c2r_direct(F[pick], n)
    scale_x = np.sqrt(np.mean(ref_x ** 2, axis=1))
    part = pick ^ 1  # the other row of each pair (rows 2p, 2p+1 share one transform)
    alone = part >= rows  # the last row of an odd count shares its transform with no row
    part = np.minimum(part, rows - 1)
    if pairing:  # a row's error is set by its pair
        other = np.sqrt(np.mean(oracle.c2r_direct(F[part], n) ** 2, axis=1))
        scale_x = np.where(alone, scale_x, np.hypot(scale_x, other))
    assert_parity(xs[pick], ref_x, n, f"small shape synthesis pairing={pairing}", scale=scale_x)
    ref_G = oracle.r2c_direct(xs[pick].astype(np.float64), mmax)
    scale_G = np.linalg.norm(xs[pick].astype(np.float64), axis=1)
    if pairing:
        other = np.linalg.norm(xs[part].astype(np.float64), axis=1)
        scale_G = np.where(alone, scale_G, np.hypot(scale_G, other))
    assert_parity(G.cpu().numpy()[pick], ref_G, mmax + 1, f"small shape analysis pairing={pairing}",
                  scale=scale_G)


# ---- band-limited real rows of any length (the any-nphi 'dft' mode) --------------------------
LAYOUTS = {"rowmajor": 1, "mmajor": 2}


def gpu_c2r(F_rowmajor, n, mmax, layout):
    m = fx()
    rows = F_rowmajor.shape[0]
    p = m.Plan(n, rows, 1, m.INVERSE, layout=LAYOUTS[layout], mmax=mmax)
    assert expected_path(n, real=True) in p.describe()
    Fin = oracle.to_mmajor(F_rowmajor) if layout == "mmajor" else F_rowmajor
    x = p.c2r(torch.from_numpy(np.ascontiguousarray(Fin, dtype=np.complex64)).cuda())
    torch.cuda.synchronize()
    p.check()
    return x.cpu().numpy()


def gpu_r2c(x, mmax, layout):
    m = fx()
    rows, n = x.shape
    p = m.Plan(n, rows, 1, m.FORWARD, layout=LAYOUTS[layout], mmax=mmax)
    assert expected_path(n, real=True) in p.describe()
    F = p.r2c(torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda())
    torch.cuda.synchronize()
    p.check()
    F = F.cpu().numpy()
    return oracle.from_mmajor(F) if layout == "mmajor" else F


REAL_LENGTHS = [3, 5, 6, 100, 999, 1000, 3000, 6000, 8191]


@pytest.mark.parametrize("n", REAL_LENGTHS)
@pytest.mark.parametrize("layout", ["rowmajor", "mmajor"])
def test_any_length_real_synthesis(n, layout, route):
    skip_same(n, route)
    for mmax in sorted({0, (n - 1) // 2, max(0, n // 7)} | ({n // 2} if n % 2 == 0 else set())):
        rows = 33 if n <= 1000 else 3
        F = wl().spectrum(7400 + n + mmax, rows, mmax)
        got = gpu_c2r(F, n, mmax, layout)
        assert_parity(got, oracle.c2r_direct(F, n), n, f"c2r n={n} mmax={mmax} {layout}")


@pytest.mark.parametrize("n", REAL_LENGTHS)
@pytest.mark.parametrize("layout", ["rowmajor", "mmajor"])
def test_any_length_real_analysis(n, layout, route):
    skip_same(n, route)
    for mmax in sorted({0, (n - 1) // 2, max(0, n // 7)} | ({n // 2} if n % 2 == 0 else set())):
        rows = 33 if n <= 1000 else 3
        x = wl().real_normal(7500 + n + mmax, rows, n)
        got = gpu_r2c(x, mmax, layout)
        ref = oracle.r2c_direct(x, mmax)
        # per-row scale ||x_row||_2 (the RMS of the full spectrum), since few bins may be kept
        scale = np.linalg.norm(x.astype(np.float64), axis=1)
        assert_parity(got, ref, mmax + 1, f"r2c n={n} mmax={mmax} {layout}", scale=scale)


@pytest.mark.parametrize("n", [1000, 6000])
def test_any_length_real_round_trip(n, route):
    mmax = (n - 1) // 2
    F = wl().spectrum(7600 + n, 4, mmax)
    x = gpu_c2r(F, n, mmax, "mmajor")
    G = gpu_r2c(x, mmax, "mmajor")
    ref = n * F.astype(np.complex128)
    ref[:, 0] = n * F[:, 0].real
    assert_parity(G, ref, mmax + 1, f"analysis(synthesis) n={n}")


# ---- lengths above 8192: the multi-pass chirp-z (four-step m-point passes over a workspace) --
# References come from the oracle's mixed-radix FFT (smallest prime factor first; a prime length
# is its direct sum), pinned to numpy: the direct O(n^2) sum of oracle.transform is too slow here.
LONG_LENGTHS = [8193, 9000, 10000, 12289, 65535, 100000, 531441, 1000000, (1 << 20) - 1]


def long_ref(x, direction, shift=False):
    if not shift:
        return oracle.fft_any(x, direction)
    if direction == -1:
        return oracle.fftshift_any(oracle.fft_any(x, -1))
    return oracle.fft_any(oracle.fftshift_any(x, 1, inverse=True), +1)


@pytest.mark.parametrize("n", LONG_LENGTHS)
@pytest.mark.parametrize("direction", [-1, 1])
def test_long_any_length_grid(n, direction, route):
    """A prime (12289), products of small primes (the mixed-radix four-step path, and forced
    onto the multi-pass chirp-z) and the largest length (m = 2^21), both directions, against
    the oracle's mixed-radix DFT."""
    skip_same(n, route)
    batch = 3 if n <= 100000 else 2
    x = wl().normal(7500 + n, batch, n)
    m = fx()
    want = "path=mixed_fourstep" if expected_path(n) == "path=mixed" else "path=bluestein_multipass"
    assert want in m.query(n, batch, 1, direction)
    got = gpu_c2c(x, n, batch, direction)
    assert_parity(got, long_ref(x, direction), n, f"long n={n} dir={direction}")


@pytest.mark.parametrize("n", [10000, 10001, 2 * 3 ** 10, 7 ** 5 * 5])
@pytest.mark.parametrize("direction", [-1, 1])
def test_long_any_length_shift_in_place(n, direction, route):
    skip_same(n, route)
    batch = 2
    x = wl().uniform(7600 + n, batch, n)
    got = gpu_c2c(x, n, batch, direction, shift=True, inplace=True)
    assert_parity(got, long_ref(x, direction, True), n, f"long shift n={n}")


def test_long_full_batch_sampled():
    """The benchmark's long any-length workload at full size (n = 100000, batch = 671: the
    mixed-radix four-step path over a 537 MB workspace), sampled rows against the oracle."""
    m = fx()
    n = 100000
    batch = (1 << 26) // n
    x = wl().tones(7350, batch, n)
    p = m.Plan(n, batch, 1, m.FORWARD)
    assert "path=mixed_fourstep" in p.describe()
    y = p.c2c(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    p.check()
    rng = np.random.default_rng(7350)
    rows = np.array(sorted({0, batch - 1, batch // 2, *rng.integers(0, batch, 9).tolist()}))
    ys = y[torch.from_numpy(rows).cuda()].cpu().numpy()
    assert_parity(ys, long_ref(x[rows], -1), n, "n=100000 full batch")


def test_long_any_length_round_trip_and_tones(route):
    n, batch = 100000, 2
    x = wl().tones(7700, batch, n)
    y = gpu_c2c(x, n, batch, -1)
    assert_parity(y, long_ref(x, -1), n, "long tones n=100000")
    z = gpu_c2c(y, n, batch, +1)
    assert_parity(z, n * x.astype(np.complex128), n, "long round trip n=100000")


@pytest.mark.parametrize("n,mmaxes", [(10000, (0, 3333, 4999, 5000)), (10001, (1, 5000)),
                                      (100000, (0, 1000)), (3 ** 9, (1, 9841))])
@pytest.mark.parametrize("layout", ["rowmajor", "mmajor"])
def test_long_real_rows(n, mmaxes, layout, route):
    """Band-limited real rows above 8192 points, two rows per transform (the mixed-radix
    four-step for lengths with prime factors 2, 3, 5, 7, and forced onto the chirp-z; the
    chirp-z otherwise), odd and even row counts, against the oracle's direct analysis and
    synthesis sums."""
    skip_same(n, route)
    for i, mmax in enumerate(mmaxes):
        rows = (3, 4)[i % 2]
        F = wl().spectrum(7800 + n + i, rows, mmax)
        got = gpu_c2r(F, n, mmax, layout)
        assert_parity(got, oracle.c2r_direct(F, n), n, f"long c2r n={n} mmax={mmax} {layout}")
        x = wl().real_normal(7900 + n + i, rows, n)
        G = gpu_r2c(x, mmax, layout)
        assert_parity(G, oracle.r2c_direct(x, mmax), mmax + 1,
                      f"long r2c n={n} mmax={mmax} {layout}",
                      scale=np.linalg.norm(x.astype(np.float64), axis=1))


@pytest.mark.parametrize("pairing", [False, True])
def test_any_length_real_large_batch_sampled(pairing):
    """Real rows of 1001 points (7 * 11 * 13: the chirp-z path) in a batch large enough for the
    radix-64 chirp-z schedule (the small batches above take the radix-16 one): sampled rows
    against the direct sums."""
    m = fx()
    n, rows, mmax = 1001, 12000, 333
    assert "radix=64x32" in m.query(n, rows, 1, m.INVERSE, m.LAYOUT_REAL_MMAJOR)
    F = wl().spectrum(7950, rows, mmax)
    syn = m.Plan(n, rows, 1, m.INVERSE, layout=m.LAYOUT_REAL_MMAJOR, mmax=mmax, pairing=pairing)
    ana = m.Plan(n, rows, 1, m.FORWARD, layout=m.LAYOUT_REAL_MMAJOR, mmax=mmax, pairing=pairing)
    x = syn.c2r(torch.from_numpy(np.ascontiguousarray(oracle.to_mmajor(F), dtype=np.complex64)).cuda())
    G = ana.r2c(x)
    torch.cuda.synchronize()
    syn.check()
    ana.check()
    pick = np.array(sorted({0, 1, rows - 2, rows - 1, *np.random.default_rng(7950).integers(0, rows, 28).tolist()}))
    xs = x.cpu().numpy()[pick]
    ref_x = oracle.c2r_direct(F[pick], n)
    scale_x = np.sqrt(np.mean(ref_x ** 2, axis=1))
    if pairing:  # a row's error is set by its pair (rows 2p, 2p+1 share one transform)
        xall = oracle.c2r_direct(F[pick ^ 1], n)
        scale_x = np.hypot(scale_x, np.sqrt(np.mean(xall ** 2, axis=1)))
    assert_parity(xs, ref_x, n, f"large real batch synthesis pairing={pairing}", scale=scale_x)
    Gs = oracle.from_mmajor(G.cpu().numpy())[pick]
    ref_G = oracle.r2c_direct(xs.astype(np.float64), mmax)
    scale_G = np.linalg.norm(xs.astype(np.float64), axis=1)
    if pairing:
        scale_G = np.hypot(scale_G, np.linalg.norm(x.cpu().numpy()[pick ^ 1].astype(np.float64), axis=1))
    assert_parity(Gs, ref_G, mmax + 1, f"large real batch analysis pairing={pairing}", scale=scale_G)
