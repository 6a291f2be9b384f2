"""Tolerances of the parity tests (GPU fp32 result vs fp64 oracle).

* rel-L2 over the whole output: ||y - y_ref||_2 / ||y_ref||_2 <= 5e-6.
* max element error per transform t:
      max_i |y_i - y_ref,i| <= 1e-5 * RMS_t(y_ref) + KAPPA * u * max_i |y_ref,i|,
  u = 2^-24 the unit roundoff of fp32.  The first term is the stated bound
  1e-5 * ||x||_2 / sqrt(N) read with the output's own scale (for a forward C2C transform
  RMS(y) = ||x||_2 by Parseval, the scale of the unitary transform).  The second term is the
  resolution of the fp32 output format at the transform's largest value: an output holding a
  spike (a tone of amplitude 1 transforms to a bin of magnitude N) cannot be stored closer than
  half an ulp of that spike, and the rounding of the last butterfly stages, made on partial sums
  of that magnitude, reaches the bins that share those butterflies at the same level.  For
  N >= 2^20 the correctly rounded fp32 value of the exact spike already misses the first term
  alone (tests/test_parity_helper.py).  For noise-like outputs max|y| is a few RMS and the
  second term is ~1e-6 RMS, so the bound stays the stated one there.

Both gates are enforced: `assert_parity` fails when either is exceeded.
"""
import json
import os

import numpy as np

REL_L2 = 5e-6
MAX_ELEM = 1e-5
U32 = 2.0 ** -24  # unit roundoff of IEEE binary32
KAPPA = 4         # fp32 ulps of the transform's largest output value


def _split(got, ref, per, scale):
    got = np.asarray(got, dtype=np.complex128 if np.iscomplexobj(got) else np.float64)
    ref = np.asarray(ref)
    err = np.abs(got - ref).reshape(-1, per)
    mag = np.abs(ref).reshape(-1, per)
    rms = np.sqrt(np.mean(mag ** 2, axis=1)) if scale is None else np.ravel(scale)
    return got, ref, err, mag, rms


def errors(got, ref, per, scale=None):
    """Return (rel_l2, worst max-element error) for transforms of `per` trailing elements.

    The second value is max over transforms of
        max_i max(|got_i - ref_i| - KAPPA * u * max|ref|, 0) / scale,
    compared directly with MAX_ELEM.  scale: per-transform error scale; default the RMS of the
    transform's reference output.
    """
    got, ref, err, mag, rms = _split(got, ref, per, scale)
    rel = float(np.linalg.norm((got - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))
    allow = KAPPA * U32 * mag.max(axis=1)
    over = np.max(np.maximum(err - allow[:, None], 0.0), axis=1)
    ratio = np.where(rms > 0, over / np.maximum(rms, 1e-300), np.where(over > 0, np.inf, 0))
    return rel, float(np.max(ratio))


def detail(got, ref, per, scale=None):
    """The plain ratio max|err| / scale (no format allowance) and the smallest allowance, in
    ulps of max|ref|, under which the 1e-5 term holds: the numbers the per-path table reports."""
    _, _, err, mag, rms = _split(got, ref, per, scale)
    raw = float(np.max(err.max(axis=1) / np.maximum(rms, 1e-300)))
    need = np.maximum(err - MAX_ELEM * rms[:, None], 0.0).max(axis=1) / np.maximum(
        U32 * mag.max(axis=1), 1e-300)
    return raw, float(np.max(need))


def assert_parity(got, ref, per, what="", scale=None):
    """Assert both gates; return (rel_l2, max-element error / scale beyond the allowance)."""
    rel, maxel = errors(got, ref, per, scale)
    log = os.environ.get("GBFFT_PARITY_LOG")
    if log:  # one JSON line per comparison, for the per-path worst-case table
        raw, need = detail(got, ref, per, scale)
        with open(log, "a") as f:
            f.write(json.dumps({"what": what, "rel_l2": rel, "max_elem": maxel,
                                "max_elem_plain": raw, "ulps_of_max_needed": need}) + "\n")
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e} > {REL_L2}"
    assert maxel <= MAX_ELEM, (f"{what}: max element error {maxel:.3e} x RMS beyond "
                               f"{KAPPA} ulps of max|y| > {MAX_ELEM} x RMS")
    return rel, maxel
