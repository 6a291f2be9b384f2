"""The allocation-free entry point fft_exec_c2c_noalloc, called through the C ABI.

It serves callers that may not allocate device memory (a host framework that owns all device
memory, latency-bound loops that cannot take cudaMalloc's implicit synchronisation); its
scratch, tables and error word are static device arrays of the library.  Each case runs two
calls in a row (the second reuses the scratch the first one left behind) and checks every
output against the fp64 oracle and against the plan-based fft_exec_c2c of the same size, within
the parity tolerance of the other tests.  The cases cover forward and inverse, the chessboard
on the forward load and on the inverse store, and in-place calls (out = in).
This file is collected last so that a stop-at-first-failure run has run everything else.
"""
import ctypes

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


def _call(L, n, batch, direction, shift, x, out, stream):
    return L.fft_exec_c2c_noalloc(n, batch, direction, shift, ctypes.c_void_p(x.data_ptr()),
                                  ctypes.c_void_p(out.data_ptr()),
                                  ctypes.c_void_p(stream.cuda_stream))


@pytest.mark.parametrize("log2n,batch,direction,shift,in_place", [
    (15, 64, -1, 1, False), (16, 2, +1, 1, False), (18, 3, +1, 0, False),
    (21, 1, -1, 0, False), (17, 4, -1, 1, True), (16, 8, +1, 1, True),
])
def test_noalloc_matches_oracle_and_plan_path_twice(log2n, batch, direction, shift, in_place):
    import fft_signal_processing_gb300 as fx
    from fft_signal_processing_gb300 import workloads

    n = 1 << log2n
    L = fx.lib()
    stream = torch.cuda.current_stream()
    plan = fx.Plan(n, batch, 1, direction, shift=bool(shift))
    for call in range(2):  # two calls in a row, different inputs
        xh = workloads.normal(700 + 10 * log2n + call, batch, n)
        x = torch.from_numpy(xh).cuda()
        ref_plan = plan.c2c(x)
        if in_place:
            out = x.clone()
            rc = _call(L, n, batch, direction, shift, out, out, stream)
        else:
            out = torch.full_like(x, float("nan"))
            rc = _call(L, n, batch, direction, shift, x, out, stream)
        assert rc == fx.FFT_OK, fx.status_string(rc)
        assert L.fft_exec_c2c_noalloc(0, 0, 0, 0, None, None,
                                      ctypes.c_void_p(stream.cuda_stream)) == fx.FFT_OK
        got = out.cpu().numpy()
        what = f"noalloc call {call} n={n} dir={direction} shift={shift} in_place={in_place}"
        assert_parity(got, oracle.transform(xh, direction, 1, bool(shift)), n, what)
        assert_parity(got, ref_plan.cpu().numpy().astype(np.complex128), n, what + " vs plan")
    plan.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import fft_signal_processing_gb300 as fx

    L = fx.lib()
    x = torch.zeros(16, dtype=torch.complex64, device="cuda")
    p = ctypes.c_void_p(x.data_ptr())
    big = fx.FFT_ERR_UNSUPPORTED_SIZE
    assert L.fft_exec_c2c_noalloc(1 << 21, 2, -1, 0, p, p, None) == big  # 2^22 points
    assert L.fft_exec_c2c_noalloc(1 << 22, 1, -1, 0, p, p, None) == big
    assert L.fft_exec_c2c_noalloc(1 << 14, 1, -1, 0, p, p, None) == big
    assert L.fft_exec_c2c_noalloc(3 << 15, 1, -1, 0, p, p, None) == big
    assert L.fft_exec_c2c_noalloc(1 << 15, 0, -1, 0, p, p, None) == fx.FFT_ERR_INVALID_ARG
    assert L.fft_exec_c2c_noalloc(1 << 15, 1, 0, 0, p, p, None) == fx.FFT_ERR_INVALID_ARG
    assert L.fft_exec_c2c_noalloc(1 << 15, 1, -1, 0, None, p, None) == fx.FFT_ERR_INVALID_ARG
    q = ctypes.c_void_p(x.data_ptr() + 8)
    assert L.fft_exec_c2c_noalloc(1 << 15, 1, -1, 0, q, p, None) == fx.FFT_ERR_MISALIGNED
    # the status form: nothing timed out
    assert L.fft_exec_c2c_noalloc(0, 0, 0, 0, None, None, None) == fx.FFT_OK
