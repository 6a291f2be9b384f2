"""GPU parity of the 1-D C2C paths (one-pass and four-step) against the fp64 oracle.

Every case runs the library through its C ABI (via the ctypes binding) on seeded inputs and
compares element by element with the oracle on the same inputs: rel-L2 <= 5e-6 and per-row
max error <= 1e-5 x the row's reference RMS (tests/parity.py); exactly where the fp32
arithmetic is exact.
"""
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


def gpu_c2c(x, n, batch, direction, shift=False, inplace=False):
    m = fx()
    p = m.Plan(n, batch, 1, direction, shift=shift)
    xd = torch.from_numpy(np.ascontiguousarray(x, dtype=np.complex64)).cuda()
    if inplace:
        p.c2c(xd, out=xd)
        y = xd
    else:
        y = p.c2c(xd)
    torch.cuda.synchronize()
    p.check()
    return y.cpu().numpy()


def rng_c64(seed, batch, n):
    from fft_signal_processing_gb300 import workloads

    return workloads.normal(seed, batch, n)


# ---- one-pass sizes: every log2 n from 0 to 14, ragged batches, both directions, shift ----
@pytest.mark.parametrize("log2n", list(range(0, 15)))
@pytest.mark.parametrize("batch", [1, 3, 67])
@pytest.mark.parametrize("direction", [-1, 1])
def test_onepass_grid(log2n, batch, direction):
    n = 1 << log2n
    x = rng_c64(1000 + log2n * 7 + batch, batch, n)
    got = gpu_c2c(x, n, batch, direction)
    assert_parity(got, oracle.transform(x, direction, 1, False), n,
                  f"n={n} batch={batch} dir={direction}")


@pytest.mark.parametrize("log2n", list(range(1, 15)))
@pytest.mark.parametrize("direction", [-1, 1])
def test_onepass_shift(log2n, direction):
    n, batch = 1 << log2n, 5
    x = rng_c64(2000 + log2n, batch, n)
    got = gpu_c2c(x, n, batch, direction, shift=True)
    assert_parity(got, oracle.transform(x, direction, 1, True), n, f"shift n={n}")


@pytest.mark.parametrize("log2n", [0, 4, 10, 12, 14])
def test_onepass_in_place(log2n):
    n, batch = 1 << log2n, 9
    x = rng_c64(3000 + log2n, batch, n)
    got = gpu_c2c(x, n, batch, -1, inplace=True)
    assert_parity(got, oracle.transform(x, -1), n, "in place")


# ---- four-step sizes 2^15 .. 2^24 ------------------------------------------------------------
@pytest.mark.parametrize("log2n", list(range(15, 25)))
@pytest.mark.parametrize("direction", [-1, 1])
def test_fourstep(log2n, direction):
    n = 1 << log2n
    batch = max(1, (1 << 21) // n) + (1 if log2n < 20 else 0)  # odd batches below 2^20
    x = rng_c64(4000 + log2n, batch, n)
    got = gpu_c2c(x, n, batch, direction)
    assert_parity(got, oracle.transform(x, direction), n, f"four-step n={n} dir={direction}")


@pytest.mark.parametrize("log2n", [15, 18, 24])
@pytest.mark.parametrize("direction", [-1, 1])
def test_fourstep_shift_and_in_place(log2n, direction):
    n, batch = 1 << log2n, 2
    x = rng_c64(5000 + log2n, batch, n)
    got = gpu_c2c(x, n, batch, direction, shift=True, inplace=True)
    assert_parity(got, oracle.transform(x, direction, 1, True), n, f"four-step shift n={n}")


# ---- the four-step path forced at one-pass sizes (GBFFT_FORCE_PATH, test override) -----------
@pytest.mark.parametrize("log2n", [12, 13, 14])
@pytest.mark.parametrize("direction", [-1, 1])
@pytest.mark.parametrize("shift", [False, True])
def test_forced_fourstep_matches_oracle(log2n, direction, shift, monkeypatch):
    """n = 2^12..2^14 planned as N1 x 256 four-step transforms (short strided columns with the
    twiddle w_n^{n2*k1} on their store, then transposed 256-point rows), compared with the
    oracle and with the default one-pass plan on the same input; normalised as well."""
    m = fx()
    n, batch = 1 << log2n, 5
    x = rng_c64(6000 + log2n + 10 * (direction > 0) + 20 * shift, batch, n)
    ref = oracle.transform(x, direction, 1, shift)
    monkeypatch.setenv("GBFFT_FORCE_PATH", "fourstep")
    p = m.Plan(n, batch, 1, direction, shift=shift)
    assert f"path=fourstep n={n}" in p.describe() and f"n1={n >> 8} n2=256" in p.describe()
    xd = torch.from_numpy(np.ascontiguousarray(x, dtype=np.complex64)).cuda()
    y = p.c2c(xd)
    p.set_normalization(True)
    yn = p.c2c(xd)
    torch.cuda.synchronize()
    p.check()
    p.close()
    assert_parity(y.cpu().numpy(), ref, n, f"forced four-step n={n} dir={direction} shift={shift}")
    assert_parity(yn.cpu().numpy(), ref / n, n, f"forced four-step normalised n={n}")
    monkeypatch.delenv("GBFFT_FORCE_PATH")
    assert_parity(gpu_c2c(x, n, batch, direction, shift), ref, n, f"one-pass n={n}")


# ---- bit-exact cases (exact fp32 arithmetic) --------------------------------------------------
@pytest.mark.parametrize("n", [1, 2, 4])
@pytest.mark.parametrize("direction", [-1, 1])
@pytest.mark.parametrize("shift", [False, True])
def test_small_integer_inputs_bit_exact(n, direction, shift):
    if shift and n == 1:
        pytest.skip("shift needs even n")
    rng = np.random.default_rng(n * 10 + (direction > 0))
    batch = 300
    x = (rng.integers(-8, 8, (batch, n)) + 1j * rng.integers(-8, 8, (batch, n))).astype(np.complex64)
    got = gpu_c2c(x, n, batch, direction, shift)
    ref = oracle.transform(x, direction, 1, shift)
    exact = np.round(ref.real) + 1j * np.round(ref.imag)  # the oracle's fp64 rounding aside
    assert np.max(np.abs(ref - exact)) < 1e-9
    np.testing.assert_array_equal(got.astype(np.complex128), exact)


@pytest.mark.parametrize("log2n", list(range(0, 25, 3)) + [12, 14, 15, 24])
def test_delta_gives_exact_ones(log2n):
    n = 1 << log2n
    x = np.zeros((2, n), np.complex64)
    x[:, 0] = 1
    got = gpu_c2c(x, n, 2, -1)
    np.testing.assert_array_equal(got, np.ones((2, n), np.complex64))
    if n >= 2:  # inverse with shift: the chessboard itself
        got = gpu_c2c(x, n, 2, 1, shift=True)
        np.testing.assert_array_equal(got.real, np.tile((-1.0) ** np.arange(n), (2, 1)))
        np.testing.assert_array_equal(got.imag, 0)


# ---- argument errors on real plans ------------------------------------------------------------
def test_exec_argument_errors():
    m = fx()
    p = m.Plan(64, 4)
    x = torch.zeros((4, 64), dtype=torch.complex64, device="cuda")
    y = torch.zeros((4, 64), dtype=torch.complex64, device="cuda")
    L = m.lib()
    import ctypes

    vp = ctypes.c_void_p
    assert L.fft_exec_c2c(p.handle, vp(0), vp(y.data_ptr()), vp(0)) == m.FFT_ERR_INVALID_ARG
    assert L.fft_exec_c2c(p.handle, vp(x.data_ptr() + 8), vp(y.data_ptr()), vp(0)) == \
        m.FFT_ERR_MISALIGNED
    # partial overlap of in and out
    assert L.fft_exec_c2c(p.handle, vp(x.data_ptr()), vp(x.data_ptr() + 64), vp(0)) == \
        m.FFT_ERR_INVALID_ARG
    # wrong exec kind
    assert L.fft_exec_r2c(p.handle, vp(x.data_ptr()), vp(y.data_ptr()), vp(0)) == \
        m.FFT_ERR_INVALID_ARG
    assert L.fft_plan_set_band_limit(p.handle, 3) == m.FFT_ERR_INVALID_ARG
    assert p.workspace_bytes() == 0
    p.check()
    with pytest.raises(TypeError):
        p.c2c(x.real.contiguous())
    big = m.Plan(1 << 16, 2)
    assert big.workspace_bytes() == 2 * (1 << 16) * 8
    assert "fourstep" in big.describe()


# ---- bounded device waits: forced timeout is reported and the context stays usable ----------
@pytest.mark.parametrize("log2n", [5, 10, 12, 13, 24])
def test_wait_timeout_reported_then_recovers(log2n):
    m = fx()
    n = 1 << log2n
    batch = 333 if log2n <= 13 else 1
    p = m.Plan(n, batch, 1, m.FORWARD)
    x = rng_c64(6000 + log2n, batch, n)
    xd = torch.from_numpy(x).cuda()
    p.set_wait_timeout(0)  # every bulk-copy wait gives up at once
    p.c2c(xd)
    with pytest.raises(m.GbfftError) as ei:
        p.check()
    assert ei.value.status == m.FFT_ERR_TIMEOUT
    p.check()  # the error word was cleared
    p.set_wait_timeout(2_000_000_000)
    y = p.c2c(xd)
    torch.cuda.synchronize()
    p.check()
    assert_parity(y.cpu().numpy(), oracle.transform(x, -1), n, "after timeout")
