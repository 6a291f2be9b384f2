"""GPU parity at the full sizes of the benchmark configurations, with the same plans (hence
the same kernels and launch geometry) the benchmark times.

* 1-D C2C N = 1024 x 64 rows, forward: every output checked.
* 1-D C2C N = 4096 x 16384 rows (512 MiB), forward with the chessboard shift, then inverse:
  sampled rows checked against the oracle (forward) and against n*x (the fp64 round trip).
* size sweep N = 2^1 .. 2^24, batch*N = 2^26 (512 MiB), 3 tones + noise per row: sampled rows
  checked against the oracle, and each sampled row's tones found at their bins.
* real rows 2048 x 4096, mmax = 1365, m-major: synthesis, then analysis, every output checked
  against the oracle's synthesis and the oracle's fp64 round trip.
* 2-D 4096 x 4096 with the (-1)^(x+y) chessboard, forward then inverse: every output checked.
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


def wl():
    from fft_signal_processing_gb300 import workloads

    return workloads


def sample_rows(batch, k, seed):
    rng = np.random.default_rng(seed)
    rows = {0, batch - 1, batch // 2}
    rows.update(rng.integers(0, batch, size=k).tolist())
    return np.array(sorted(rows))


def test_c2c_1024x64_full():
    m = fx()
    x = wl().uniform(11, 64, 1024)
    p = m.Plan(1024, 64, 1, m.FORWARD)
    y = p.c2c(torch.from_numpy(x).cuda()).cpu().numpy()
    assert_parity(y, oracle.transform(x, -1), 1024, "1024 x 64")


def test_c2c_4096x16384_shift_round_trip():
    m = fx()
    n, batch = 4096, 16384
    x = wl().normal(12, batch, n)
    fwd = m.Plan(n, batch, 1, m.FORWARD, shift=True)
    inv = m.Plan(n, batch, 1, m.INVERSE, shift=True)
    xd = torch.from_numpy(x).cuda()
    y = fwd.c2c(xd)
    z = inv.c2c(y)
    torch.cuda.synchronize()
    fwd.check()
    rows = sample_rows(batch, 61, 12)
    rt = torch.from_numpy(rows).cuda()
    ys, zs = y[rt].cpu().numpy(), z[rt].cpu().numpy()
    xs = x[rows]
    assert_parity(ys, oracle.transform(xs, -1, 1, True), n, "4096 forward+shift")
    assert_parity(zs, oracle.transform(oracle.transform(xs, -1, 1, True), +1, 1, True), n,
                  "4096 round trip")


@pytest.mark.parametrize("log2n", list(range(1, 25)))
def test_size_sweep_full_batch(log2n):
    m = fx()
    n = 1 << log2n
    batch = (1 << 26) // n
    x = wl().tones(13 + log2n, batch, n)
    p = m.Plan(n, batch, 1, m.FORWARD)
    y = p.c2c(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    p.check()
    rows = sample_rows(batch, 5 if n >= (1 << 20) else 29, 13 + log2n)
    ys = y[torch.from_numpy(rows).cuda()].cpu().numpy()
    ref = oracle.transform(x[rows], -1)
    assert_parity(ys, ref, n, f"sweep n={n}")
    f, phi = wl().tone_params(13 + log2n, batch, n)
    for i, r in enumerate(rows):  # unit tones land on their bins with magnitude ~ n
        for k in set(f[r]):
            amp = n * abs(np.sum(np.exp(1j * phi[r][f[r] == k])))
            # the N(0, 0.1) noise adds about 0.1 * sqrt(2n) at any bin: allow 6 sigma
            assert abs(abs(ys[i, k]) - amp) < 0.05 * n + 0.6 * (2 * n) ** 0.5


def test_real_2048x4096_mmajor_round_trip():
    m = fx()
    n, rows, mmax = 4096, 2048, 1365
    F = wl().spectrum(14, rows, mmax)
    syn = m.Plan(n, rows, 1, m.INVERSE, layout=m.LAYOUT_REAL_MMAJOR, mmax=mmax)
    ana = m.Plan(n, rows, 1, m.FORWARD, layout=m.LAYOUT_REAL_MMAJOR, mmax=mmax)
    Fd = torch.from_numpy(np.ascontiguousarray(oracle.to_mmajor(F))).cuda()
    x = syn.c2r(Fd)
    G = ana.r2c(x)
    torch.cuda.synchronize()
    syn.check()
    xr = oracle.c2r(F, n)
    assert_parity(x.cpu().numpy(), xr, n, "real synthesis")
    assert_parity(oracle.from_mmajor(G.cpu().numpy()), oracle.r2c(xr, mmax), mmax + 1,
                  "real round trip")


def test_2d_4096_shift_round_trip():
    m = fx()
    n = 4096
    img = wl().image(15, 1, n)
    fwd = m.Plan(n, 1, 2, m.FORWARD, shift=True)
    inv = m.Plan(n, 1, 2, m.INVERSE, shift=True)
    y = fwd.c2c(torch.from_numpy(img).cuda())
    z = inv.c2c(y)
    torch.cuda.synchronize()
    fwd.check()
    ref = oracle.transform(img, -1, 2, True)
    assert_parity(y.cpu().numpy(), ref, n * n, "2-D forward+shift")
    assert_parity(z.cpu().numpy(), oracle.transform(ref, +1, 2, True), n * n, "2-D round trip")
