"""GPU parity of the band-limited real-row path (R2C analysis / C2R synthesis, row-major and
m-major spectra) and of the 2-D path, against the fp64 oracle."""
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


LAYOUTS = {"rowmajor": 1, "mmajor": 2}


def gpu_c2r(F_rowmajor, n, mmax, layout):
    m = fx()
    rows = F_rowmajor.shape[0]
    p = m.Plan(n, rows, 1, m.INVERSE, layout=LAYOUTS[layout], mmax=mmax)
    Fin = oracle.to_mmajor(F_rowmajor) if layout == "mmajor" else F_rowmajor
    Fd = torch.from_numpy(np.ascontiguousarray(Fin, dtype=np.complex64)).cuda()
    x = p.c2r(Fd)
    torch.cuda.synchronize()
    return x.cpu().numpy()


def gpu_r2c(x, mmax, layout):
    m = fx()
    rows, n = x.shape
    p = m.Plan(n, rows, 1, m.FORWARD, layout=LAYOUTS[layout], mmax=mmax)
    F = p.r2c(torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda())
    torch.cuda.synchronize()
    F = F.cpu().numpy()
    return oracle.from_mmajor(F) if layout == "mmajor" else F


def mmax_cases(n):
    h = n // 2
    return sorted({0, h - 1, max(0, h // 3), max(0, (2 * h) // 3)})


@pytest.mark.parametrize("log2n", list(range(2, 16)))
@pytest.mark.parametrize("layout", ["rowmajor", "mmajor"])
def test_c2r_grid(log2n, layout):
    n = 1 << log2n
    for mmax in mmax_cases(n):
        # odd row counts take the direct-load path, even ones the tensor-copy path (m-major)
        rows = (67 if mmax % 2 else 64) if n <= 4096 else (5 if mmax % 2 else 6)
        F = wl().spectrum(100 + log2n, rows, mmax)
        got = gpu_c2r(F, n, mmax, layout)
        assert_parity(got, oracle.c2r(F, n), n, f"c2r n={n} mmax={mmax} {layout}")


@pytest.mark.parametrize("log2n", list(range(2, 16)))
@pytest.mark.parametrize("layout", ["rowmajor", "mmajor"])
def test_r2c_grid(log2n, layout):
    n = 1 << log2n
    for mmax in mmax_cases(n):
        rows = (67 if mmax % 2 else 64) if n <= 4096 else (5 if mmax % 2 else 6)
        x = wl().real_normal(200 + log2n, rows, n)
        got = gpu_r2c(x, mmax, layout)
        ref = oracle.r2c(x, mmax)
        # per-row error scale: the RMS of the row's full spectrum, ||x_row||_2 (Parseval),
        # since few bins may be kept
        assert_parity(got, ref, mmax + 1, f"r2c n={n} mmax={mmax} {layout}",
                      scale=np.linalg.norm(x.astype(np.float64), axis=1))


@pytest.mark.parametrize("layout", ["rowmajor", "mmajor"])
def test_real_n4_bit_exact(layout):
    """n = 4: every twiddle is 0 or +-1 and every product exact, so the Hermitian assembly,
    the two-for-one recombination and the spectrum layout must match bit for bit."""
    rng = np.random.default_rng(7)
    rows, n, mmax = 131, 4, 1
    F = (rng.integers(-8, 8, (rows, 2)) + 1j * rng.integers(-8, 8, (rows, 2))).astype(np.complex64)
    x = gpu_c2r(F, n, mmax, layout)
    ref = oracle.c2r(F, n)
    np.testing.assert_array_equal(x.astype(np.float64), np.round(ref))
    xr = rng.integers(-8, 8, (rows, n)).astype(np.float32)
    G = gpu_r2c(xr, mmax, layout)
    refG = oracle.r2c(xr, mmax)
    np.testing.assert_array_equal(G.astype(np.complex128),
                                  np.round(refG.real) + 1j * np.round(refG.imag))


@pytest.mark.parametrize("layout", ["rowmajor", "mmajor"])
def test_real_roundtrip(layout):
    n, rows, mmax = 1024, 33, 341
    F = wl().spectrum(300, rows, mmax)
    x = gpu_c2r(F, n, mmax, layout)
    G = gpu_r2c(x, mmax, layout)
    ref = oracle.r2c(oracle.c2r(F, n), mmax)  # the fp64 round trip of F
    assert_parity(G, ref, mmax + 1, f"real round trip {layout}")


def test_real_argument_errors():
    m = fx()
    p = m.Plan(64, 4, 1, m.FORWARD, layout=1)
    assert p.mmax == 31
    L = m.lib()
    assert L.fft_plan_set_band_limit(p.handle, 33) == m.FFT_ERR_INVALID_ARG  # above n/2
    assert L.fft_plan_set_band_limit(p.handle, -1) == m.FFT_ERR_INVALID_ARG
    x = torch.zeros((4, 64), dtype=torch.float32, device="cuda")
    import ctypes

    vp = ctypes.c_void_p
    assert L.fft_exec_c2r(p.handle, vp(x.data_ptr()), vp(x.data_ptr()), vp(0)) == \
        m.FFT_ERR_INVALID_ARG  # forward plan run as synthesis
    assert L.fft_exec_r2c(p.handle, vp(x.data_ptr()), vp(x.data_ptr()), vp(0)) == \
        m.FFT_ERR_INVALID_ARG  # in and out overlap
    assert L.fft_exec_c2c(p.handle, vp(x.data_ptr()), vp(x.data_ptr()), vp(0)) == \
        m.FFT_ERR_INVALID_ARG


# ---- 2-D -------------------------------------------------------------------------------------
def gpu_2d(img, direction, shift, inplace=False):
    m = fx()
    batch, n, _ = img.shape
    p = m.Plan(n, batch, 2, direction, shift=shift)
    xd = torch.from_numpy(np.ascontiguousarray(img, dtype=np.complex64)).cuda()
    y = p.c2c(xd, out=xd) if inplace else p.c2c(xd)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("log2n", list(range(1, 13)))
@pytest.mark.parametrize("direction", [-1, 1])
@pytest.mark.parametrize("shift", [False, True])
def test_2d_grid(log2n, direction, shift):
    n = 1 << log2n
    batch = 3 if n <= 512 else 1
    img = wl().image(400 + log2n, batch, n)
    got = gpu_2d(img, direction, shift, inplace=(log2n % 2 == 0))
    assert_parity(got, oracle.transform(img, direction, 2, shift), n * n,
                  f"2d n={n} dir={direction} shift={shift}")


def test_2d_small_integer_bit_exact():
    rng = np.random.default_rng(11)
    for n in (2, 4):
        img = (rng.integers(-4, 4, (7, n, n)) + 1j * rng.integers(-4, 4, (7, n, n))).astype(np.complex64)
        for direction in (-1, 1):
            for shift in (False, True):
                got = gpu_2d(img, direction, shift)
                ref = oracle.transform(img, direction, 2, shift)
                exact = np.round(ref.real) + 1j * np.round(ref.imag)
                np.testing.assert_array_equal(got.astype(np.complex128), exact)


# ---- bounded waits of the 2-D and large-N kernels: forced timeout, then a correct run -----
@pytest.mark.parametrize("n,dims,batch", [(1024, 2, 1), (4096, 2, 1), (1 << 16, 1, 2),
                                          (1 << 23, 1, 1)])
def test_wait_timeout_column_and_transposed_kernels(n, dims, batch):
    m = fx()
    p = m.Plan(n, batch, dims, m.FORWARD)
    shape = (batch, n, n) if dims == 2 else (batch, n)
    x = wl().normal(900 + dims, batch * (n if dims == 2 else 1), n).reshape(shape)
    xd = torch.from_numpy(x).cuda()
    p.set_wait_timeout(0)
    p.c2c(xd)
    with pytest.raises(m.GbfftError) as ei:
        p.check()
    assert ei.value.status == m.FFT_ERR_TIMEOUT
    p.set_wait_timeout(2_000_000_000)
    y = p.c2c(xd)
    torch.cuda.synchronize()
    p.check()
    ref = oracle.transform(x, -1, dims, False)
    assert_parity(y.cpu().numpy(), ref, n * n if dims == 2 else n, "after timeout")


def test_wait_timeout_real_synthesis():
    m = fx()
    n, rows, mmax = 4096, 64, 1365
    p = m.Plan(n, rows, 1, m.INVERSE, layout=LAYOUTS["mmajor"], mmax=mmax)
    F = wl().spectrum(950, rows, mmax)
    Fd = torch.from_numpy(np.ascontiguousarray(oracle.to_mmajor(F))).cuda()
    p.set_wait_timeout(0)
    p.c2r(Fd)
    with pytest.raises(m.GbfftError) as ei:
        p.check()
    assert ei.value.status == m.FFT_ERR_TIMEOUT
    p.set_wait_timeout(2_000_000_000)
    x = p.c2r(Fd)
    torch.cuda.synchronize()
    p.check()
    assert_parity(x.cpu().numpy(), oracle.c2r(F, n), n, "after timeout")


def test_wait_timeout_real_analysis():
    """The persistent analysis kernel (m-major spectrum, even row count) waits on bulk copies of
    its real rows: a forced timeout is reported, and the next run is correct."""
    m = fx()
    n, rows, mmax = 4096, 64, 1365
    p = m.Plan(n, rows, 1, m.FORWARD, layout=LAYOUTS["mmajor"], mmax=mmax)
    x = wl().real_normal(960, rows, n)
    xd = torch.from_numpy(x).cuda()
    p.set_wait_timeout(0)
    p.r2c(xd)
    with pytest.raises(m.GbfftError) as ei:
        p.check()
    assert ei.value.status == m.FFT_ERR_TIMEOUT
    p.set_wait_timeout(2_000_000_000)
    F = p.r2c(xd)
    torch.cuda.synchronize()
    p.check()
    assert_parity(oracle.from_mmajor(F.cpu().numpy()), oracle.r2c(x, mmax), mmax + 1,
                  "analysis after timeout", scale=np.linalg.norm(x.astype(np.float64), axis=1))


# ---- the Nyquist bin: mmax = n/2, the full n/2 + 1 half spectrum -----------------------------
@pytest.mark.parametrize("n", [4, 8, 64, 4096, 1 << 15, 1000, 6000])
@pytest.mark.parametrize("layout", ["rowmajor", "mmajor"])
@pytest.mark.parametrize("rows", [7, 64])  # odd: direct loads/stores; even: tensor copies
def test_nyquist_full_half_spectrum(n, layout, rows):
    h = n // 2
    if n > 4096:
        rows = 3 if rows == 7 else 4
    x = wl().real_normal(300 + n + rows, rows, n)
    F = gpu_r2c(x, h, layout)
    ref = oracle.r2c_direct(x, h) if n & (n - 1) else oracle.r2c(x, h)
    assert_parity(F, ref, h + 1, f"r2c Nyquist n={n} {layout}",
                  scale=np.linalg.norm(x.astype(np.float64), axis=1))
    assert np.all(F[:, h].imag == 0)  # real Nyquist bin
    G = wl().spectrum(400 + n + rows, rows, h)
    got = gpu_c2r(G, n, h, layout)
    refx = oracle.c2r_direct(G, n) if n & (n - 1) else oracle.c2r(G, n)
    assert_parity(got, refx, n, f"c2r Nyquist n={n} {layout}")


def test_band_limit_range():
    m = fx()
    p = m.Plan(16, 2, 1, m.FORWARD, layout=1)
    L = m.lib()
    assert L.fft_plan_set_band_limit(p.handle, 8) == m.FFT_OK  # n/2: Nyquist
    assert L.fft_plan_set_band_limit(p.handle, 9) == m.FFT_ERR_INVALID_ARG
    assert L.fft_plan_set_band_limit(p.handle, -1) == m.FFT_ERR_INVALID_ARG
    q = m.Plan(15, 2, 1, m.FORWARD, layout=1)  # odd length: 2*mmax <= n means mmax <= 7
    assert L.fft_plan_set_band_limit(q.handle, 7) == m.FFT_OK
    assert L.fft_plan_set_band_limit(q.handle, 8) == m.FFT_ERR_INVALID_ARG


# ---- rectangular 2-D images (fft_plan_create_2d) ----------------------------------------------
@pytest.mark.parametrize("ny,nx", [(4096, 2), (2, 4096), (64, 128), (128, 64), (1024, 256),
                                   (4096, 8), (8, 4096), (4096, 16), (512, 4096), (32, 2)])
@pytest.mark.parametrize("direction", [-1, 1])
@pytest.mark.parametrize("shift", [False, True])
def test_2d_rectangular(ny, nx, direction, shift):
    m = fx()
    batch = 2 if ny * nx <= (1 << 20) else 1
    rng = np.random.default_rng(ny * 7 + nx)
    img = (rng.standard_normal((batch, ny, nx)) +
           1j * rng.standard_normal((batch, ny, nx))).astype(np.complex64)
    p = m.Plan(nx, batch, 2, direction, shift=shift, ny=ny)
    assert f"n={ny}x{nx}" in p.describe()
    xd = torch.from_numpy(img).cuda()
    y = p.c2c(xd, out=xd) if (ny + nx) % 3 == 0 else p.c2c(xd)  # some in place
    torch.cuda.synchronize()
    p.check()
    assert_parity(y.cpu().numpy(), oracle.transform(img, direction, 2, shift), nx * ny,
                  f"2d {ny}x{nx} dir={direction} shift={shift}")
