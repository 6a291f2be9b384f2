"""The parity gates themselves (CPU).

Each gate must reject an output just outside its bound and accept one just inside, so that a
GPU test that passes has met both bounds.  The fp32-format allowance of the max-element gate
(KAPPA ulps of the transform's largest output) is pinned to things independent of this
library: the correctly rounded fp32 value of the exact (fp64 oracle) transform, and the fp32
FFT of another implementation (torch's CPU FFT), on the spiky outputs of the tone and
plane-wave workloads.
"""
import numpy as np
import pytest

import oracle
import parity
from parity import KAPPA, MAX_ELEM, REL_L2, U32, assert_parity, detail, errors


def _rows(seed=0, rows=64, n=4096):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((rows, n)) + 1j * rng.standard_normal((rows, n))


def _allow(ref_row):
    return KAPPA * U32 * np.abs(ref_row).max()


def test_one_element_over_the_max_element_bound_fails():
    ref = _rows()
    rms = np.sqrt(np.mean(np.abs(ref[5]) ** 2))
    got = ref.copy()
    got[5, 17] += 2e-5 * rms  # 2x the bound, far inside the rel-L2 gate
    rel, maxel = errors(got, ref, ref.shape[1])
    assert rel < REL_L2
    assert maxel == pytest.approx((2e-5 * rms - _allow(ref[5])) / rms, rel=1e-9)
    assert maxel > 1.8e-5  # the format allowance is ~1e-6 RMS on noise-like rows
    with pytest.raises(AssertionError, match="max element"):
        assert_parity(got, ref, ref.shape[1])


def test_one_element_inside_the_max_element_bound_passes():
    ref = _rows(1)
    rms = np.sqrt(np.mean(np.abs(ref[9]) ** 2))
    got = ref.copy()
    got[9, 4000] -= 9e-6j * rms
    rel, maxel = assert_parity(got, ref, ref.shape[1])
    assert maxel <= 9e-6
    assert detail(got, ref, ref.shape[1])[0] == pytest.approx(9e-6, rel=1e-9)


def test_rel_l2_gate_fails_on_spread_error():
    ref = _rows(2, rows=8, n=1024)
    got = ref * (1 + 8e-6)  # every element off by 8e-6 relative: rel-L2 8e-6 > 5e-6
    with pytest.raises(AssertionError, match="rel-L2"):
        assert_parity(got, ref, ref.shape[1])


def test_explicit_scale_is_used():
    ref = np.ones((2, 8))
    got = ref.copy()
    got[1, 3] += 3e-6
    _, maxel = errors(got, ref, 8, scale=np.array([1.0, 0.1]))
    assert maxel == pytest.approx((3e-6 - KAPPA * U32) / 0.1)
    with pytest.raises(AssertionError):
        assert_parity(got, ref, 8, scale=np.array([1.0, 0.1]))


def test_zero_reference_row_needs_exact_zero():
    ref = np.zeros((2, 4))
    assert errors(ref.copy(), ref, 4)[1] == 0.0
    got = ref.copy()
    got[0, 0] = 1e-30
    assert errors(got, ref, 4)[1] == np.inf


def _tones(log2n, rows=2):
    from fft_signal_processing_gb300 import workloads

    x = workloads.tones(1, rows, 1 << log2n)
    return x, oracle.transform(x, -1)


def test_correctly_rounded_spike_misses_the_plain_bound():
    """At N = 2^20 a unit tone gives a bin of magnitude 2^20; its correctly rounded fp32 value
    is already further from the exact one than 1e-5 RMS, so no fp32 output meets the plain
    bound there.  The same rounded result passes with the format allowance."""
    x, ref = _tones(20)
    rounded = ref.astype(np.complex64).astype(np.complex128)
    plain, need = detail(rounded, ref, x.shape[1])
    assert plain > MAX_ELEM
    assert need <= 1.0  # within one ulp of the largest output
    assert_parity(rounded, ref, x.shape[1], "rounded exact 2^20")


def test_independent_fp32_fft_needs_and_meets_the_allowance():
    """torch's CPU fp32 FFT (a different implementation) on the tone rows and on a plane-wave
    image: it misses the plain bound, and meets it with the allowance."""
    torch = pytest.importorskip("torch")
    from fft_signal_processing_gb300 import workloads

    x, ref = _tones(20)
    got = torch.fft.fft(torch.from_numpy(x)).numpy()
    assert detail(got, ref, x.shape[1])[0] > MAX_ELEM
    assert_parity(got, ref, x.shape[1], "torch fp32 2^20 tones")
    img = workloads.image(5, 1, 1024)
    ref2 = oracle.transform(img, -1, 2)
    got2 = torch.fft.fft2(torch.from_numpy(img)).numpy()
    assert detail(got2, ref2, 1024 * 1024)[0] > MAX_ELEM
    assert_parity(got2, ref2, 1024 * 1024, "torch fp32 1024^2 image")


def test_allowance_still_catches_a_wrong_bin_next_to_a_spike():
    """A single wrong output next to the spike, 2e-6 of the spike's magnitude (8x the format
    allowance, too small for the rel-L2 gate), fails although the row holds a spike."""
    x, ref = _tones(16, rows=1)
    got = ref.astype(np.complex64).astype(np.complex128)
    k = int(np.argmax(np.abs(ref[0])))
    got[0, (k + 1) % x.shape[1]] += 2e-6 * np.abs(ref[0, k])
    assert errors(got, ref, x.shape[1])[0] < REL_L2
    with pytest.raises(AssertionError, match="max element"):
        assert_parity(got, ref, x.shape[1])


def test_allowance_is_negligible_on_noise_like_rows():
    ref = _rows(3, rows=4, n=1 << 16)
    for r in ref:
        assert _allow(r) / np.sqrt(np.mean(np.abs(r) ** 2)) < 0.15 * MAX_ELEM
    assert parity.KAPPA == 4
