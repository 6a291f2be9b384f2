"""Distinct plans used concurrently from several host threads (the header's thread-safety
statement): in a fresh process, threads make the first launches of the same kernels at the same
time (the launchers' per-device set-up runs under a lock), each on its own stream, and every
result must match the fp64 oracle."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import sys, threading
    sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
    import numpy as np, torch
    import fft_signal_processing_gb300 as fx
    from fft_signal_processing_gb300 import workloads
    import oracle
    from parity import assert_parity
    torch.cuda.init()
    cases = [(4096, 64, 1), (1 << 16, 4, 1), (1000, 32, 1), (2048, 2, 2), (512, 64, 1)] * 2
    start = threading.Barrier(len(cases))
    errors = []
    def work(i, n, batch, dims):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            shape = (batch, n, n) if dims == 2 else (batch, n)
            x = workloads.normal(3000 + i, batch * (n if dims == 2 else 1), n).reshape(shape)
            with torch.cuda.stream(s):
                xd = torch.from_numpy(x).cuda()
                p = fx.Plan(n, batch, dims, fx.FORWARD)
                start.wait()  # every thread makes its first launch at once
                y = p.c2c(xd, stream=s)
            s.synchronize()
            p.check()
            assert_parity(y.cpu().numpy(), oracle.transform(x, -1, dims), n * n if dims == 2 else n,
                          f"thread {{i}} n={{n}}")
            p.close()
        except Exception as e:
            errors.append(repr(e))
    ts = [threading.Thread(target=work, args=(i, *c)) for i, c in enumerate(cases)]
    [t.start() for t in ts]
    [t.join() for t in ts]
    print("ERRORS", errors)
    sys.exit(1 if errors else 0)
""")


@pytest.fixture(scope="module", autouse=True)
def built():
    import __graft_entry__

    __graft_entry__.build()


def test_concurrent_first_launches_from_host_threads():
    code = SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
