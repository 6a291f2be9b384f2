"""Tolerances of the parity tests (GPU fp32 result vs fp64 oracle).

* rel-L2 over the whole output: ||y - y_ref||_2 / ||y_ref||_2 <= 5e-6.
* max element error per transform: max_i |y_i - y_ref,i| <= 1e-5 * ||y_ref||_2 / sqrt(len),
  i.e. 1e-5 times the RMS of that transform's reference output.  For a forward C2C transform
  the RMS of the output equals ||x||_2 (Parseval), so this is the bound
  max|err| <= 1e-5 * ||x||_2 written with the output's own scale.
"""
import numpy as np

REL_L2 = 5e-6
MAX_ELEM = 1e-5


def errors(got, ref, per, scale=None):
    """Return (rel_l2, worst max-element ratio) with transforms of `per` trailing elements.

    scale: per-transform error scale; default the RMS of the transform's reference output.
    """
    got = np.asarray(got, dtype=np.complex128 if np.iscomplexobj(got) else np.float64)
    ref = np.asarray(ref)
    rel = float(np.linalg.norm((got - ref).ravel()) / max(np.linalg.norm(ref.ravel()), 1e-300))
    g = (got - ref).reshape(-1, per)
    r = ref.reshape(-1, per)
    rms = np.sqrt(np.mean(np.abs(r) ** 2, axis=1)) if scale is None else np.ravel(scale)
    maxerr = np.max(np.abs(g), axis=1)
    ratio = np.where(rms > 0, maxerr / np.maximum(rms, 1e-300), np.where(maxerr > 0, np.inf, 0))
    return rel, float(np.max(ratio)) * 1.0


def assert_parity(got, ref, per, what="", scale=None):
    rel, ratio = errors(got, ref, per, scale)
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e} > {REL_L2}"
    assert ratio <= 1.0, (f"{what}: max element error {ratio * MAX_ELEM:.3e} x RMS "
                          f"> {MAX_ELEM} x RMS")
    return rel, ratio * MAX_ELEM
