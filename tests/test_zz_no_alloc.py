"""The allocation-free entry point fft_exec_c2c_noalloc, called through the C ABI.

It serves callers that may not allocate device memory (a host framework that owns all device
memory, latency-bound loops that cannot take cudaMalloc's implicit synchronisation); its
scratch and tables are static device arrays of the library.  Its output must equal that of
the plan-based fft_exec_c2c of the same size, within the parity tolerance of the other tests,
on two calls in a row (the second call reuses the scratch the first one left behind).
This file is collected last so that a stop-at-first-failure run has run everything else.
"""
import ctypes

import numpy as np
import pytest

from parity import assert_parity

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__

    __graft_entry__.build()


@pytest.mark.parametrize("log2n,batch,direction,shift", [
    (15, 64, -1, 1), (18, 3, +1, 0), (21, 1, -1, 0),
])
def test_noalloc_matches_plan_path_twice(log2n, batch, direction, shift):
    import fft_signal_processing_gb300 as fx
    from fft_signal_processing_gb300 import workloads

    n = 1 << log2n
    L = fx.lib()
    stream = torch.cuda.current_stream()
    plan = fx.Plan(n, batch, 1, direction, shift=bool(shift))
    for call in range(2):  # two calls in a row, different inputs
        x = torch.from_numpy(workloads.normal(700 + 10 * log2n + call, batch, n)).cuda()
        ref = plan.c2c(x)
        out = torch.full_like(x, float("nan"))
        rc = L.fft_exec_c2c_noalloc(n, batch, direction, shift, ctypes.c_void_p(x.data_ptr()),
                                    ctypes.c_void_p(out.data_ptr()),
                                    ctypes.c_void_p(stream.cuda_stream))
        assert rc == fx.FFT_OK, fx.status_string(rc)
        torch.cuda.synchronize()
        assert_parity(out.cpu().numpy(), ref.cpu().numpy().astype(np.complex128), n,
                      f"noalloc call {call} n={n}")
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
