"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every function
declared in include/gbfft.h, and the planner validates its arguments and picks its paths."""
import ctypes
import os
import re

import pytest

import fft_signal_processing_gb300 as fx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbfft.h")


@pytest.fixture(scope="module", autouse=True)
def built():
    from fft_signal_processing_gb300 import _build

    _build.build()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fft_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(fx.ABI_SYMBOLS)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(fx.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version():
    for st in (0, -1, -2, -3, -4, -5, -6, -7):
        assert fx.status_string(st).startswith("FFT_")
    assert fx.status_string(fx.FFT_ERR_BOUNDS).startswith("FFT_ERR_BOUNDS")
    assert fx.status_string(-99) == "unknown status"
    assert fx.lib().fft_version() >= 10000


def test_destroy_null_is_ok():
    assert fx.lib().fft_plan_destroy(None) == fx.FFT_OK


def q(n, batch=1, dims=1, direction=-1, layout=0, shift=0):
    return fx.lib().fft_plan_query(n, batch, dims, direction, layout, shift, None, 0)


@pytest.mark.parametrize("n", [0, -4, (1 << 20) + 1, 3 << 20, 1000003 * 3])
def test_lengths_outside_the_supported_set_rejected(n):
    assert q(n) == fx.FFT_ERR_UNSUPPORTED_SIZE


@pytest.mark.parametrize("n,m", [(11, 32), (13 * 3, 128), (1001, 2048), (1025, 4096),
                                 (4096 + 1, 16384), (8191, 16384)])
def test_any_length_rows_take_the_chirp_z_path(n, m):
    """Lengths with a prime factor above 7 (11, 13, 1001 = 7*11*13, 1025 = 25*41, 4097,
    8191) take the one-pass chirp-z kernel."""
    d = fx.query(n, 5)
    assert "path=bluestein" in d and f"m={m} " in d and "kernels=1" in d
    assert m >= 2 * n - 1 and m // 2 < 2 * n - 1  # the smallest power of two that suffices
    assert q(n, shift=1) == fx.FFT_OK  # odd lengths too: the shift is a complex exponential
    # band-limited real rows of these lengths take the same path; 2-D images stay powers of two
    d = fx.query(n, 5, layout=2, direction=1)
    assert "path=bluestein" in d and f"mmax={(n - 1) // 2} " in d and "synthesis" in d
    assert q(n, dims=2) == fx.FFT_ERR_UNSUPPORTED_SIZE


@pytest.mark.parametrize("n,radix", [(3, "3"), (5, "5"), (6, "3x2"), (12, "3x4"), (100, "5x5x4"),
                                     (1000, "5x5x5x8"), (3000, "5x5x5x3x8"), (6561, "3x" * 7 + "3"),
                                     (7168, "7x8x8x8x2"), (8000, "5x5x5x8x8")])
def test_smooth_lengths_take_the_mixed_radix_path(n, radix, monkeypatch):
    """Lengths up to 8192 whose prime factors are 2, 3, 5 and 7 take the mixed-radix kernel
    (radices 7, 5, 3 first, then 8s and a last 4 or 2), complex and real, shift allowed;
    GBFFT_FORCE_PATH=chirpz sends them to the chirp-z kernel instead."""
    d = fx.query(n, 5)
    assert "path=mixed" in d and f"radix={radix} " in d and "kernels=1" in d
    assert q(n, shift=1) == fx.FFT_OK
    d = fx.query(n, 6, layout=2, direction=1)
    assert "path=mixed" in d and f"mmax={(n - 1) // 2} " in d and "synthesis" in d
    monkeypatch.setenv("GBFFT_FORCE_PATH", "chirpz")
    assert "path=bluestein" in fx.query(n, 5)
    assert "path=bluestein" in fx.query(n, 5, layout=1)


@pytest.mark.parametrize("n,n1,n2", [(9000, 90, 100), (10000, 100, 100), (49152, 192, 256),
                                      (100000, 250, 400), (531441, 243, 2187),
                                      (823543, 343, 2401), (1000000, 500, 2000)])
def test_long_smooth_lengths_take_the_mixed_fourstep_path(n, n1, n2, monkeypatch):
    """Rows above 8192 points whose prime factors are 2, 3, 5, 7 take two mixed-radix passes
    (real rows two per transform, the analysis with a third, unpack pass), split n = N1*N2
    with N1 the largest divisor up to min(512, sqrt(n)) that leaves N2 <= 8192; the forced
    chirp-z route takes the multi-pass chirp-z path."""
    d = fx.query(n, 3)
    assert "path=mixed_fourstep" in d and f"n1={n1} n2={n2} " in d and "kernels=2" in d
    assert n1 * n2 == n and n1 <= 512 and n2 <= 8192 and n1 * n1 <= n
    assert q(n, shift=1) == fx.FFT_OK
    d = fx.query(n, 3, layout=1)
    assert "path=mixed_fourstep" in d and "rows_per_transform=2" in d and "kernels=3" in d
    d = fx.query(n, 3, layout=2, direction=1)
    assert "path=mixed_fourstep" in d and "synthesis" in d and "kernels=2" in d
    monkeypatch.setenv("GBFFT_FORCE_PATH", "chirpz")
    assert "path=bluestein_multipass" in fx.query(n, 3)
    assert "path=bluestein_multipass" in fx.query(n, 3, layout=1)


@pytest.mark.parametrize("n,m", [(8193, 1 << 15), (12289, 1 << 15), (16385, 1 << 16),
                                 (100003, 1 << 18), ((1 << 20) - 1, 1 << 21)])
def test_long_any_length_rows_take_the_multipass_chirp_z_path(n, m):
    d = fx.query(n, 3)
    assert "path=bluestein_multipass" in d and f"m={m} " in d and "kernels=6" in d
    l = m.bit_length() - 1
    assert f"n1={1 << (l // 2)} n2={1 << (l - l // 2)}" in d
    d = fx.query(n, 3, layout=1)
    assert "path=bluestein_multipass" in d and "rows_per_transform=2" in d


def test_size_limits():
    assert q(1 << 24) == fx.FFT_OK
    assert q(1 << 25) == fx.FFT_ERR_UNSUPPORTED_SIZE
    assert q(1 << 12, dims=2) == fx.FFT_OK
    assert q(1 << 13, dims=2) == fx.FFT_ERR_UNSUPPORTED_SIZE
    assert q(1, dims=2) == fx.FFT_ERR_UNSUPPORTED_SIZE
    assert q(1 << 15, layout=1) == fx.FFT_OK
    assert q(1 << 16, layout=1) == fx.FFT_ERR_UNSUPPORTED_SIZE
    assert q(2, layout=1) == fx.FFT_ERR_UNSUPPORTED_SIZE


@pytest.mark.parametrize("args", [
    dict(batch=0), dict(batch=-1), dict(dims=3), dict(direction=0), dict(direction=2),
    dict(layout=3), dict(shift=2), dict(layout=1, shift=1), dict(layout=2, dims=2),
])
def test_invalid_arguments(args):
    assert q(64, **args) == fx.FFT_ERR_INVALID_ARG


def test_shift_needs_even_n():
    assert q(1, shift=1) == fx.FFT_ERR_INVALID_ARG
    assert q(2, shift=1) == fx.FFT_OK


def test_batch_overflow_rejected():
    assert q(1 << 20, batch=1 << 40) == fx.FFT_ERR_UNSUPPORTED_SIZE


def test_create_rejects_before_touching_the_device():
    h = ctypes.c_void_p(1)
    rc = fx.lib().fft_plan_create((1 << 20) + 1, 1, 1, -1, 0, 0, ctypes.byref(h))
    assert rc == fx.FFT_ERR_UNSUPPORTED_SIZE and not h.value
    assert fx.lib().fft_plan_create(8, 1, 1, -1, 0, 0, None) == fx.FFT_ERR_INVALID_ARG


def test_null_plan_calls():
    L = fx.lib()
    assert L.fft_plan_set_band_limit(None, 1) == fx.FFT_ERR_INVALID_ARG
    assert L.fft_plan_set_real_pairing(None, 1) == fx.FFT_ERR_INVALID_ARG
    assert L.fft_plan_workspace_bytes(None, None) == fx.FFT_ERR_INVALID_ARG
    assert L.fft_plan_describe(None, None, 0) == fx.FFT_ERR_INVALID_ARG
    assert L.fft_exec_c2c(None, None, None, None) == fx.FFT_ERR_INVALID_ARG
    assert L.fft_exec_r2c(None, None, None, None) == fx.FFT_ERR_INVALID_ARG
    assert L.fft_exec_c2r(None, None, None, None) == fx.FFT_ERR_INVALID_ARG
    assert L.fft_plan_check(None) == fx.FFT_ERR_INVALID_ARG


@pytest.mark.parametrize("n,path,radix", [
    (1, "onepass", "1"), (16, "onepass", "16"), (64, "onepass", "8x8"), (1024, "onepass", "32x32"),
    (2048, "onepass", "64x32"), (4096, "onepass", "64x64"), (8192, "onepass", "32x16x16"),
    (1 << 14, "onepass", "32x32x16"), (1 << 15, "fourstep", None), (1 << 22, "fourstep", None),
    (1 << 23, "fourstep", None), (1 << 24, "fourstep", None),
])
def test_path_choice(n, path, radix):
    d = fx.query(n, 4)
    assert f"path={path}" in d
    if radix:
        assert f"radix={radix} " in d
    l = n.bit_length() - 1
    if path == "fourstep":
        assert f"n1={1 << (l // 2)} n2={1 << (l - l // 2)}" in d


def test_checked_build_links_and_exports_every_symbol():
    """The checked variant (-DGBFFT_CHECKED) builds from the same sources and exports the same
    ABI; its GPU behaviour is covered by tests/test_gpu_checked.py."""
    import ctypes
    from fft_signal_processing_gb300 import _build

    path = _build.build(checked=True)
    assert path.endswith("libgbfft_checked.so")
    L = ctypes.CDLL(path)
    for name in fx.ABI_SYMBOLS:
        assert hasattr(L, name), name


def test_forced_path_override(monkeypatch):
    """GBFFT_FORCE_PATH (test override, read at each plan creation or query): "fourstep" plans
    C2C rows of 2^12..2^14 points as N1 x 256 four-step transforms and changes nothing else;
    "onepass" or an empty value keeps the default; any other value is an argument error."""
    monkeypatch.setenv("GBFFT_FORCE_PATH", "fourstep")
    for l in (12, 13, 14):
        d = fx.query(1 << l, 3)
        assert "path=fourstep" in d and f"n1={1 << (l - 8)} n2=256" in d
    assert "path=onepass" in fx.query(2048, 3)
    assert f"n1={1 << 7} n2={1 << 8}" in fx.query(1 << 15, 3)
    assert "path=2d" in fx.query(4096, 1, dims=2)
    assert "path=real" in fx.query(4096, 8, layout=2, direction=1)
    assert "path=mixed" in fx.query(1000, 3)
    for v in ("onepass", "default", ""):
        monkeypatch.setenv("GBFFT_FORCE_PATH", v)
        assert "path=onepass" in fx.query(4096, 3)
        assert "path=mixed" in fx.query(1000, 3)
    monkeypatch.setenv("GBFFT_FORCE_PATH", "chirpz")
    assert "path=bluestein" in fx.query(1000, 3) and "path=onepass" in fx.query(4096, 3)
    monkeypatch.setenv("GBFFT_FORCE_PATH", "four-step")
    assert q(4096) == fx.FFT_ERR_INVALID_ARG
    monkeypatch.delenv("GBFFT_FORCE_PATH")
    assert "path=onepass" in fx.query(4096, 3)


def test_2d_and_real_paths():
    assert "path=2d" in fx.query(4096, 1, dims=2, shift=True)
    d = fx.query(4096, 2048, layout=2, direction=1)
    assert "path=real" in d and "core=2048" in d and "mmajor" in d


def test_shift_argument_errors_before_touching_the_device():
    L = fx.lib()
    p = ctypes.c_void_p
    assert L.fft_shift(None, p(4096), 4, 1, 1, 1, 0, None) == fx.FFT_ERR_INVALID_ARG
    assert L.fft_shift(p(4096), p(4096), 5, 1, 1, 1, 0, None) == fx.FFT_ERR_INVALID_ARG  # odd in place
    assert L.fft_shift(p(4096), p(4096), 4, 3, 1, 2, 0, None) == fx.FFT_ERR_INVALID_ARG  # odd ny in place
    assert L.fft_shift(p(4096), p(1 << 20), 4, 2, 1, 1, 0, None) == fx.FFT_ERR_INVALID_ARG  # dims 1, ny != 1
    assert L.fft_shift(p(4096), p(4104), 4, 1, 1, 1, 0, None) == fx.FFT_ERR_INVALID_ARG  # overlap
    assert L.fft_shift(p(4096), p(1 << 20), 4, 1, 1, 3, 0, None) == fx.FFT_ERR_INVALID_ARG  # dims
    assert L.fft_shift(p(4096), p(1 << 20), 4, 1, 1, 1, 2, None) == fx.FFT_ERR_INVALID_ARG  # inverse
    assert L.fft_shift(p(4100), p(1 << 20), 4, 1, 1, 1, 0, None) == fx.FFT_ERR_MISALIGNED
    assert L.fft_shift(p(4096), p(1 << 20), 1 << 40, 2, 1, 2, 0, None) == fx.FFT_ERR_UNSUPPORTED_SIZE


@pytest.mark.parametrize("ny,nx", [(4096, 2), (2, 4096), (64, 128), (4096, 8), (8, 4096)])
def test_rectangular_2d_plans(ny, nx):
    d = fx.query(nx, 3, dims=2, ny=ny)
    assert f"path=2d n={ny}x{nx} " in d and "kernels=2" in d
    L = fx.lib()
    assert L.fft_plan_query_2d(nx, 3 * ny, 1, -1, 0, None, 0) == fx.FFT_ERR_UNSUPPORTED_SIZE
    assert L.fft_plan_query_2d(nx, 0, 1, -1, 0, None, 0) == fx.FFT_ERR_UNSUPPORTED_SIZE
    assert L.fft_plan_query_2d(nx, 8192, 1, -1, 0, None, 0) == fx.FFT_ERR_UNSUPPORTED_SIZE
    assert L.fft_plan_create_2d(nx, ny, 1, -1, 0, None) == fx.FFT_ERR_INVALID_ARG


def test_every_smooth_length_plans_a_valid_mixed_schedule():
    """Every length up to 2^20 whose prime factors are 2, 3, 5 and 7 (and is not a power of
    two) plans the mixed-radix path: one pass up to 8192 points with radices from
    {2, 3, 4, 5, 7, 8} whose product is n (odd radices first, then 8s and one 4 or 2), the
    four-step above with n1*n2 = n, n1 <= min(512, sqrt(n)), n2 <= 8192 and both factors
    scheduled the same way; every other length takes a chirp-z path."""
    def smooth(v):
        for f in (2, 3, 5, 7):
            while v % f == 0:
                v //= f
        return v == 1

    def check_radix(text, m):
        rs = [int(r) for r in text.split("x")]
        prod = 1
        for r in rs:
            prod *= r
        assert prod == m and all(r in (2, 3, 4, 5, 7, 8) for r in rs) and len(rs) <= 16
        odd = [r for r in rs if r % 2]
        assert rs[:len(odd)] == odd  # odd radices first
        even = rs[len(odd):]
        assert all(r == 8 for r in even[:-1]) and even.count(4) + even.count(2) <= 1

    seen = 0
    for n in range(3, (1 << 20) + 1):
        if n & (n - 1) == 0 or not smooth(n):
            continue
        d = fx.query(n, 2)
        seen += 1
        if n <= 8192:
            assert "path=mixed " in d, (n, d)
            check_radix(d.split("radix=")[1].split()[0], n)
        else:
            assert "path=mixed_fourstep" in d, (n, d)
            n1 = int(d.split("n1=")[1].split()[0])
            n2 = int(d.split("n2=")[1].split()[0])
            assert n1 * n2 == n and n1 <= 512 and n1 * n1 <= n and n2 <= 8192, (n, n1, n2)
            check_radix(d.split("pass1=columns(radix=")[1].split()[0], n1)
            check_radix(d.split("pass2=rows_transposed(radix=")[1].split()[0], n2)
    assert seen > 1000
    for n in (11, 13 * 8, 1001, 8191, 8193, 12289, 99991):
        assert "path=bluestein" in fx.query(n, 2)
