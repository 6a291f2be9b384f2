"""Bit-exact tests of the load and store epilogues (the index-only paths).

With the index-only diagnostic (fft_plan_set_diagnostic) a plan's kernels skip every butterfly,
twiddle and recombination, so each value travels through the production kernels' load and store
epilogues alone: the chessboard sign flips, the four-step transposed store, the Hermitian gather
of a synthesis, the pack and unpack of two real rows per transform, and the row-major and
m-major spectrum layouts.  On small-integer inputs every operation left is exact, so the outputs
must equal the oracle's index maps bit for bit (compared with ==, so -0 == +0), at the sizes the
hook is built for: 4096 points and 2^15 points.
"""
import numpy as np
import pytest

import oracle

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


def ints(seed, shape, complex_=True):
    rng = np.random.default_rng(seed)
    a = rng.integers(-64, 64, shape).astype(np.float64)
    if complex_:
        a = a + 1j * rng.integers(-64, 64, shape)
    return a


def same(got, ref):
    np.testing.assert_array_equal(np.asarray(got).astype(np.complex128 if np.iscomplexobj(got) else np.float64),
                                  np.asarray(ref))


@pytest.mark.parametrize("log2n,n1", [(12, None), (15, 1 << 7)])
@pytest.mark.parametrize("direction", [-1, 1])
@pytest.mark.parametrize("shift", [False, True])
def test_c2c_epilogues(log2n, n1, direction, shift):
    """One-pass 4096 points: y = x, or the chessboard (-1)^j on the forward load / inverse
    store.  Four-step 2^15 points: the transposed store X[k1 + N1*k2] of the [N1][N2]
    intermediate, with the chessboard on the first pass's load or the second pass's store."""
    m = fx()
    n, batch = 1 << log2n, 6
    x = ints(100 + log2n, (batch, n))
    p = m.Plan(n, batch, 1, direction, shift=shift)
    p.set_index_only(True)
    y = p.c2c(torch.from_numpy(x.astype(np.complex64)).cuda()).cpu().numpy()
    p.check()
    p.close()
    ref = x
    if shift and direction == -1:
        ref = oracle.chessboard(ref)
    if n1:
        ref = oracle.fourstep_order(ref, n1)
    if shift and direction == 1:
        ref = oracle.chessboard(ref)
    same(y, ref)


def real_plans(n, rows, mmax, layout, pairing):
    m = fx()
    syn = m.Plan(n, rows, 1, m.INVERSE, layout=LAYOUTS[layout], mmax=mmax, pairing=pairing)
    ana = m.Plan(n, rows, 1, m.FORWARD, layout=LAYOUTS[layout], mmax=mmax, pairing=pairing)
    syn.set_index_only(True)
    ana.set_index_only(True)
    return syn, ana


@pytest.mark.parametrize("log2n", [12, 15])
@pytest.mark.parametrize("layout", ["rowmajor", "mmajor"])
@pytest.mark.parametrize("rows", [6, 5])  # even m-major row counts take the tensor-copy path
def test_real_epilogues(log2n, layout, rows):
    """n/2-point real path.  Synthesis: the gathered X_0..X_{n/2-1} (X_0 = Re F_0, zero above
    mmax) written as x_{2k} = Re X_k, x_{2k+1} = Im X_k.  Analysis: the real row read as
    z_k = x_{2k} + i x_{2k+1} and scattered as F_m = z_{m mod n/2}, m <= mmax, into the
    layout."""
    n = 1 << log2n
    h = n // 2
    for mmax in (h - 1, h, h // 3):
        syn, ana = real_plans(n, rows, mmax, layout, False)
        F = ints(200 + log2n + mmax, (rows, mmax + 1))
        Fin = oracle.to_mmajor(F) if layout == "mmajor" else F
        x = syn.c2r(torch.from_numpy(np.ascontiguousarray(Fin).astype(np.complex64)).cuda())
        x = x.cpu().numpy()
        X = oracle.hermitian_half(F, n)
        ref = np.empty((rows, n))
        ref[:, 0::2], ref[:, 1::2] = X.real, X.imag
        same(x, ref)
        xr = ints(300 + log2n + mmax, (rows, n), complex_=False)
        G = ana.r2c(torch.from_numpy(xr.astype(np.float32)).cuda()).cpu().numpy()
        G = oracle.from_mmajor(G) if layout == "mmajor" else G
        z = xr[:, 0::2] + 1j * xr[:, 1::2]
        same(G, z[:, np.arange(mmax + 1) % h])
        for p in (syn, ana):
            p.check()
            p.close()


@pytest.mark.parametrize("layout", ["rowmajor", "mmajor"])
@pytest.mark.parametrize("rows", [6, 5])
def test_real_pair_epilogues(layout, rows):
    """Two rows per transform, 4096 points.  Synthesis: x1 = Re Y, x2 = Im Y of the packed
    Hermitian spectrum Y = X1 + i X2.  Analysis: the unpack of the packed row y = x1 + i x2
    itself (X1 = (y_k + conj y_{n-k})/2, X2 = (y_k - conj y_{n-k})/(2i)), in the layout."""
    n, h = 4096, 2048
    for mmax in (h - 1, h, 700):
        syn, ana = real_plans(n, rows, mmax, layout, True)
        F = ints(400 + mmax, (rows, mmax + 1))
        Fin = oracle.to_mmajor(F) if layout == "mmajor" else F
        x = syn.c2r(torch.from_numpy(np.ascontiguousarray(Fin).astype(np.complex64)).cuda())
        Y = oracle.pair_assemble(F, n)
        ref = np.empty((2 * Y.shape[0], n))
        ref[0::2], ref[1::2] = Y.real, Y.imag
        same(x.cpu().numpy(), ref[:rows])
        xr = ints(500 + mmax, (rows, n), complex_=False)
        G = ana.r2c(torch.from_numpy(xr.astype(np.float32)).cuda()).cpu().numpy()
        G = oracle.from_mmajor(G) if layout == "mmajor" else G
        same(G, oracle.pair_unpack(oracle.pair_pack(xr), mmax, rows))
        for p in (syn, ana):
            p.check()
            p.close()


def test_index_only_is_refused_elsewhere():
    m = fx()
    L = m.lib()
    for n in (2048, 1 << 16, 1000):
        p = m.Plan(n, 2)
        assert L.fft_plan_set_diagnostic(p.handle, 1) == m.FFT_ERR_UNSUPPORTED_SIZE
        p.close()
    p = m.Plan(4096, 2)
    assert L.fft_plan_set_diagnostic(p.handle, 7) == m.FFT_ERR_INVALID_ARG
    assert L.fft_plan_set_diagnostic(p.handle, 1) == m.FFT_OK
    assert L.fft_plan_set_diagnostic(p.handle, 0) == m.FFT_OK
    p.close()
