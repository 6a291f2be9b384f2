"""GPU parity of the standalone fftshift / ifftshift (fft_shift, index rotation) against the
oracle's rotation, bit for bit (pure data movement): rows of odd and even lengths, square and
rectangular images, out of place in both directions, in place for even extents, and the
benchmark's full-size workload (16384 rows of 4096 points, 512 MiB)."""
import numpy as np
import pytest

import oracle

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


def run(x, dims, inverse, inplace=False, offset=0):
    xd = torch.from_numpy(x).cuda()
    if offset:  # an 8-byte-aligned (not 16) start: the single-point path
        buf = torch.empty(x.size + 1, dtype=torch.complex64, device="cuda")
        buf[1:] = xd.reshape(-1)
        xd = buf[1:].reshape(x.shape)
    out = xd if inplace else None
    y = fx().shift(xd, dims=dims, inverse=inverse, out=out)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("n", [1, 2, 3, 7, 8, 62, 1000, 1001, 4096])
@pytest.mark.parametrize("inverse", [False, True])
def test_rows(n, inverse):
    x = data(n, 37, n)
    ref = oracle.fftshift_any(x, 1, inverse).astype(np.complex64)
    np.testing.assert_array_equal(run(x, 1, inverse), ref)
    np.testing.assert_array_equal(run(x, 1, inverse, offset=1), ref)
    if n % 2 == 0:
        np.testing.assert_array_equal(run(x, 1, inverse, inplace=True), ref)


@pytest.mark.parametrize("ny,nx", [(4, 4), (5, 7), (8, 6), (6, 10), (33, 64), (1024, 1024)])
@pytest.mark.parametrize("inverse", [False, True])
def test_images(ny, nx, inverse):
    x = data(ny * 1000 + nx, 3, ny, nx)
    ref = oracle.fftshift_any(x, 2, inverse).astype(np.complex64)
    np.testing.assert_array_equal(run(x, 2, inverse), ref)
    if nx % 2 == 0 and ny % 2 == 0:
        np.testing.assert_array_equal(run(x, 2, inverse, inplace=True), ref)


def test_round_trip_odd():
    x = data(5, 9, 7, 13)
    y = run(x, 2, False)
    np.testing.assert_array_equal(run(y, 2, True), x)


def test_full_size_rows():
    n, batch = 4096, 16384
    x = data(11, batch, n)
    y = run(x, 1, False)
    np.testing.assert_array_equal(y, np.roll(x, n // 2, axis=-1))  # numpy's rotation, full size
