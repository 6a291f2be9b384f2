"""The checked build (libgbfft_checked.so, compiled with -DGBFFT_CHECKED): the copy-engine
kernels test each run-time index of a global access and each tensor-copy coordinate against the
extent of its buffer or tensor, record FFT_ERR_BOUNDS and skip the access if one falls outside.

In a fresh process that loads the checked library (GBFFT_CHECKED=1), one case per kernel family
runs through the C ABI: every plan must report FFT_OK from fft_plan_check (no index check
failed) and every output must match the fp64 oracle within the parity tolerance.  Families:
bulk-copy rows (2^6, 2^12), long rows (2^13, 2^14), column tiles and transposed rows of the
four-step path (2^15, with the shift), the big tile kernels (2^22 and a 4096 x 4096 image), the
per-tile and persistent real-row kernels (odd and even row counts, row-major and m-major
spectra, the Nyquist bin, 2^15-point rows), the multi-pass chirp-z with the filter on the column
load, and the allocation-free entry point.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import ctypes, sys
    sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
    import numpy as np, torch
    import fft_signal_processing_gb300 as fx
    from fft_signal_processing_gb300 import workloads
    import oracle
    from parity import assert_parity
    assert fx.LIB_PATH.endswith("libgbfft_checked.so"), fx.LIB_PATH
    L = fx.lib()
    maps = open("/proc/self/maps").read()
    assert "libgbfft_checked.so" in maps and "libgbfft.so" not in maps

    def c2c(n, batch, direction, shift=False, dims=1, seed=1):
        shape = (batch, n, n) if dims == 2 else (batch, n)
        x = workloads.normal(seed, batch * (n if dims == 2 else 1), n).reshape(shape)
        p = fx.Plan(n, batch, dims, direction, shift=shift)
        y = p.c2c(torch.from_numpy(x).cuda())
        p.check()  # raises GbfftError(FFT_ERR_BOUNDS) if an index check failed
        p.close()
        assert_parity(y.cpu().numpy(), oracle.transform(x, direction, dims, shift),
                      n * n if dims == 2 else n, f"checked c2c n={{n}} dims={{dims}}")

    def real(n, rows, mmax, layout, seed):
        lay = fx.LAYOUT_REAL_MMAJOR if layout == "mmajor" else fx.LAYOUT_REAL_ROWMAJOR
        F = workloads.spectrum(seed, rows, mmax)
        Fin = oracle.to_mmajor(F) if layout == "mmajor" else F
        syn = fx.Plan(n, rows, 1, fx.INVERSE, layout=lay, mmax=mmax)
        x = syn.c2r(torch.from_numpy(np.ascontiguousarray(Fin, dtype=np.complex64)).cuda())
        syn.check()
        syn.close()
        ref = oracle.c2r(F, n)
        assert_parity(x.cpu().numpy(), ref, n, f"checked c2r n={{n}} rows={{rows}}")
        ana = fx.Plan(n, rows, 1, fx.FORWARD, layout=lay, mmax=mmax)
        G = ana.r2c(x)
        ana.check()
        ana.close()
        G = G.cpu().numpy()
        G = oracle.from_mmajor(G) if layout == "mmajor" else G
        assert_parity(G, oracle.r2c(ref, mmax), mmax + 1, f"checked r2c n={{n}} rows={{rows}}")

    c2c(64, 67, -1, seed=2)
    c2c(4096, 33, +1, shift=True, seed=3)
    c2c(8192, 5, -1, seed=4)
    c2c(1 << 14, 3, +1, shift=True, seed=5)
    c2c(1 << 15, 3, -1, shift=True, seed=6)
    c2c(1 << 15, 2, +1, shift=True, seed=7)
    c2c(1 << 22, 1, -1, seed=8)
    c2c(4096, 1, -1, shift=True, dims=2, seed=9)
    real(4096, 2048, 1365, "mmajor", 10)   # persistent kernels
    real(4096, 7, 2048, "mmajor", 11)      # odd rows: per-tile kernels, Nyquist bin
    real(4096, 6, 2048, "rowmajor", 12)
    real(1 << 15, 4, 1 << 14, "mmajor", 13)

    n, rows = 100000, 2                    # multi-pass chirp-z (filter on the column load)
    x = workloads.normal(14, rows, n)
    p = fx.Plan(n, rows, 1, fx.FORWARD)
    y = p.c2c(torch.from_numpy(x).cuda())
    p.check()
    p.close()
    assert_parity(y.cpu().numpy(), oracle.fft_any(x, -1), n, "checked chirp-z n=100000")

    n, batch = 1 << 16, 2                  # allocation-free entry point
    x = torch.from_numpy(workloads.normal(15, batch, n)).cuda()
    out = torch.empty_like(x)
    s = torch.cuda.current_stream()
    rc = L.fft_exec_c2c_noalloc(n, batch, -1, 1, ctypes.c_void_p(x.data_ptr()),
                                ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(s.cuda_stream))
    assert rc == fx.FFT_OK, fx.status_string(rc)
    rc = L.fft_exec_c2c_noalloc(0, 0, -1, 0, None, None, ctypes.c_void_p(s.cuda_stream))
    assert rc == fx.FFT_OK, fx.status_string(rc)
    assert_parity(out.cpu().numpy(), oracle.transform(x.cpu().numpy(), -1, 1, True), n,
                  "checked noalloc")
    print("CHECKED OK")
""")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__
    from fft_signal_processing_gb300 import _build

    __graft_entry__.build()
    _build.build(checked=True)


def test_checked_build_reports_no_index_error_and_matches_oracle():
    code = SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    env = dict(os.environ, GBFFT_CHECKED="1")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=900, env=env)
    assert r.returncode == 0 and "CHECKED OK" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
