"""GPU parity of the real-row option that packs two real rows into one complex transform
(Mota, "High Performance Fourier Transforms on GPUs with GLSL", §2.6 Eq. 17-18), for
power-of-two rows (n-point complex core) and for rows of other lengths (chirp-z path), against
the fp64 oracle's analysis and synthesis."""
import numpy as np
import pytest

import oracle
from parity import assert_parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

LAYOUTS = {"rowmajor": 1, "mmajor": 2}


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


def c2r(F, n, mmax, layout):
    m = fx()
    p = m.Plan(n, F.shape[0], 1, m.INVERSE, layout=LAYOUTS[layout], mmax=mmax, pairing=True)
    assert "rows_per_transform=2" in p.describe()
    Fin = oracle.to_mmajor(F) if layout == "mmajor" else F
    x = p.c2r(torch.from_numpy(np.ascontiguousarray(Fin, dtype=np.complex64)).cuda())
    torch.cuda.synchronize()
    p.close()
    return x.cpu().numpy()


def r2c(x, mmax, layout):
    m = fx()
    rows, n = x.shape
    p = m.Plan(n, rows, 1, m.FORWARD, layout=LAYOUTS[layout], mmax=mmax, pairing=True)
    F = p.r2c(torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda())
    torch.cuda.synchronize()
    p.close()
    F = F.cpu().numpy()
    return oracle.from_mmajor(F) if layout == "mmajor" else F


def mmax_cases(n):
    h = n // 2
    return sorted({0, max(0, h - 1), h, max(0, h // 3)})


def pair_scale(per_row):
    """Error scale of rows transformed two at a time: the RMS of the packed transform's output,
    sqrt(s1^2 + s2^2) for the pair's per-row scales s1, s2 (a row paired with the zero row
    keeps its own).  Rounding in the packed transform is relative to the pair as a whole, so a
    row far smaller than its partner carries an error set by the partner."""
    s = np.asarray(per_row, dtype=np.float64)
    out = s.copy()
    for p in range(0, len(s) - 1, 2):
        out[p] = out[p + 1] = np.hypot(s[p], s[p + 1])
    return out


def check_both(n, rows, mmax, layout, seed, direct):
    F = wl().spectrum(seed, rows, mmax)
    ref_x = oracle.c2r_direct(F, n) if direct else oracle.c2r(F, n)
    assert_parity(c2r(F, n, mmax, layout), ref_x, n,
                  f"pair c2r n={n} rows={rows} mmax={mmax} {layout}",
                  scale=pair_scale(np.sqrt(np.mean(ref_x ** 2, axis=1))))
    x = wl().real_normal(seed + 1, rows, n)
    ref_F = oracle.r2c_direct(x, mmax) if direct else oracle.r2c(x, mmax)
    assert_parity(r2c(x, mmax, layout), ref_F, mmax + 1,
                  f"pair r2c n={n} rows={rows} mmax={mmax} {layout}",
                  scale=pair_scale(np.linalg.norm(x.astype(np.float64), axis=1)))


@pytest.mark.parametrize("log2n", list(range(2, 15)))
@pytest.mark.parametrize("layout", ["rowmajor", "mmajor"])
def test_pair_power_of_two_grid(log2n, layout):
    n = 1 << log2n
    for i, mmax in enumerate(mmax_cases(n)):
        rows = (67, 64, 5, 6)[i % 4] if n <= 4096 else (3, 4)[i % 2]  # odd and even batches
        check_both(n, rows, mmax, layout, 500 + 10 * log2n + i, direct=False)


@pytest.mark.parametrize("n", [3, 5, 12, 100, 1000, 1001, 4097, 8191])
@pytest.mark.parametrize("layout", ["rowmajor", "mmajor"])
def test_pair_any_length(n, layout):
    for i, mmax in enumerate(sorted({0, n // 3, (n - 1) // 2, n // 2})):
        rows = (33, 8)[i % 2]
        check_both(n, rows, mmax, layout, 700 + n + i, direct=True)


@pytest.mark.parametrize("layout", ["rowmajor", "mmajor"])
def test_pair_n4_bit_exact(layout):
    """n = 4: every twiddle is 0 or +-1 and the packing, unpacking, Hermitian assembly and the
    spectrum layout are exact on small integers (the halving in the unpack included), so the
    results must match bit for bit, for an odd number of rows."""
    rng = np.random.default_rng(11)
    rows, n, mmax = 131, 4, 2
    F = (rng.integers(-8, 8, (rows, 3)) + 1j * rng.integers(-8, 8, (rows, 3))).astype(np.complex64)
    x = c2r(F, n, mmax, layout)
    np.testing.assert_array_equal(x.astype(np.float64), np.round(oracle.c2r(F, n)))
    xr = rng.integers(-8, 8, (rows, n)).astype(np.float32)
    G = r2c(xr, mmax, layout)
    ref = oracle.r2c(xr, mmax)
    np.testing.assert_array_equal(G.astype(np.complex128), np.round(ref.real) + 1j * np.round(ref.imag))


def test_pair_matches_one_row_path_full_size():
    """The real workload (2048 rows x 4096, mmax = 1365, m-major): pairing and the n/2-point
    path agree with the oracle on the same inputs."""
    m = fx()
    n, rows, mmax = 4096, 2048, 1365
    F = wl().spectrum(4, rows, mmax)
    Fd = torch.from_numpy(np.ascontiguousarray(oracle.to_mmajor(F), dtype=np.complex64)).cuda()
    ref = oracle.c2r(F, n)
    for pairing in (False, True):
        syn = m.Plan(n, rows, 1, m.INVERSE, layout=m.LAYOUT_REAL_MMAJOR, mmax=mmax, pairing=pairing)
        ana = m.Plan(n, rows, 1, m.FORWARD, layout=m.LAYOUT_REAL_MMAJOR, mmax=mmax, pairing=pairing)
        x = syn.c2r(Fd)
        G = ana.r2c(x)
        torch.cuda.synchronize()
        assert_parity(x.cpu().numpy(), ref, n, f"pairing={pairing} synthesis")
        assert_parity(oracle.from_mmajor(G.cpu().numpy()), oracle.r2c(ref, mmax), mmax + 1,
                      f"pairing={pairing} analysis(synthesis)")
        syn.close()
        ana.close()


def test_pairing_arguments():
    m = fx()
    L = m.lib()
    p = m.Plan(64, 4)  # C2C plan
    assert L.fft_plan_set_real_pairing(p.handle, 1) == m.FFT_ERR_INVALID_ARG
    q = m.Plan(1 << 15, 2, 1, m.FORWARD, layout=m.LAYOUT_REAL_ROWMAJOR)
    assert L.fft_plan_set_real_pairing(q.handle, 1) == m.FFT_ERR_UNSUPPORTED_SIZE
    r = m.Plan(1 << 14, 2, 1, m.FORWARD, layout=m.LAYOUT_REAL_ROWMAJOR)
    assert L.fft_plan_set_real_pairing(r.handle, 2) == m.FFT_ERR_INVALID_ARG
    assert L.fft_plan_set_real_pairing(r.handle, 1) == m.FFT_OK
    assert L.fft_plan_set_real_pairing(r.handle, 0) == m.FFT_OK
    for x in (p, q, r):
        x.close()
