"""GPU parity of normalised plans (fft_plan_set_normalization): the output scaled by 1/n
(1/(nx*ny) for images), Mota's inverse scaling ("High Performance Fourier Transforms on GPUs
with GLSL", §2.2 Eq. 5 and §2.7), on every path: the small-row, bulk-copy and long-row
one-pass kernels, both four-step variants, square and rectangular images, and the chirp-z
path; the normalised inverse undoes the forward transform."""
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


def data(seed, *shape):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(shape) + 1j * rng.standard_normal(shape)).astype(np.complex64)


CASES = [  # (n, batch, ny or None)
    (16, 33, None), (1024, 9, None), (8192, 3, None), (1 << 16, 2, None), (1 << 22, 1, None),
    (1000, 5, None), (1001, 5, None), (64, 2, 64), (4096, 1, 4096), (4096, 1, 8),
]


@pytest.mark.parametrize("n,batch,ny", CASES)
@pytest.mark.parametrize("direction", [-1, 1])
@pytest.mark.parametrize("shift", [False, True])
def test_normalised_output(n, batch, ny, direction, shift):
    m = fx()
    dims = 1 if ny is None else 2
    shape = (batch, n) if dims == 1 else (batch, ny, n)
    x = data(n + (ny or 0) + batch, *shape)
    p = m.Plan(n, batch, dims, direction, shift=shift, ny=ny, normalize=True)
    y = p.c2c(torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    p.check()
    size = n * (ny or 1)
    ref = oracle.transform(x, direction, dims, shift) / size
    assert_parity(y.cpu().numpy(), ref, size, f"normalised n={n} ny={ny}")


@pytest.mark.parametrize("n", [4096, 1000, 1 << 18])
def test_normalised_inverse_undoes_forward(n):
    m = fx()
    x = data(n, 3, n)
    f = m.Plan(n, 3, 1, m.FORWARD, shift=True)
    i = m.Plan(n, 3, 1, m.INVERSE, shift=True, normalize=True)
    z = i.c2c(f.c2c(torch.from_numpy(x).cuda()))
    torch.cuda.synchronize()
    assert_parity(z.cpu().numpy(), x.astype(np.complex128), n, f"round trip n={n}")
    i.set_normalization(False)  # and back: unnormalised again (n * x)
    z = i.c2c(f.c2c(torch.from_numpy(x).cuda()))
    torch.cuda.synchronize()
    assert_parity(z.cpu().numpy(), n * x.astype(np.complex128), n, f"unnormalised n={n}")


def test_normalization_arguments():
    m = fx()
    L = m.lib()
    assert L.fft_plan_set_normalization(None, 1) == m.FFT_ERR_INVALID_ARG
    p = m.Plan(64, 2, 1, m.FORWARD)
    assert L.fft_plan_set_normalization(p.handle, 2) == m.FFT_ERR_INVALID_ARG
    r = m.Plan(64, 2, 1, m.FORWARD, layout=1)
    assert L.fft_plan_set_normalization(r.handle, 1) == m.FFT_ERR_INVALID_ARG  # real layouts
