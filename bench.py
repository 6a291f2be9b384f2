"""Benchmark of the batched fp32 FFT library on one node, one process per GPU.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step is one pass of the whole path over one batch of synthetic, seeded input already
resident in HBM.  The default workload is the batched 1-D C2C round trip: N = 4096 points,
16384 rows (512 MiB of complex64), a forward transform with the fftshift folded in as the
(-1)^j chessboard on its load, then the inverse transform (chessboard on its store) -- two
kernel launches per step.  Other workloads (--workload): c2c_1024 (N = 1024 x 64 rows, forward),
sweep_<log2n> (batch*N = 2^26 rows of 3 tones + noise, forward), any_<n> (the same for a
length n <= 2^20 that is not a power of two: the mixed-radix path for lengths with prime
factors 2, 3, 5, 7 only, else the chirp-z path), realany_<n> (the real
workload below for such a length, mmax = n/3; realanypair_<n>: two rows per transform), real
(2048 rows x 4096, mmax = 1365, synthesis then analysis, m-major spectrum; realpair: two rows
per transform), 2d (4096 x 4096, forward with the 2-D
chessboard then inverse), shift_<n> (standalone fftshift of 2^26 points in rows of n; this one
reports GB/s, as it moves data and computes nothing).

Metric: effective GFLOP/s = 5*N*log2(N) per complex transform (2.5*N*log2(N) per real row,
2 * 5*n^2*log2(n) per 2-D image) / time, whole job over all ranks.  The JSON line also carries
the minimum-traffic HBM GB/s of the step (16 bytes per complex point per read+write pass) and
the roofline of the dominant kernel, measured live with CUDA events on the launching stream.

--impl reference runs the fp64 CPU oracle instead (the deliberately slow baseline of this
library), on a bounded sample of the same workload, on the host cores.

Timing rules: W >= 3 untimed warm-up steps; K timed steps bracketed by a barrier and a device
synchronisation, the K-step window repeated (the same count on every rank) until --min-seconds
(default 1 s) has passed, the median per-step time reported; inputs are larger than L2 for the
default workload (smaller ones flush L2 between steps by writing a 512 MiB buffer, outside the
timed kernel windows); nvidia-smi clocks are sampled during the timed region.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="c2c_4096")
    ap.add_argument("--impl", default="gbfft", choices=["gbfft", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="repeat the K-step timed window until about this long has passed")
    ap.add_argument("--rows", type=int, default=0,
                    help="override the batch per GPU (small profiling captures only)")
    return ap.parse_args()


# ---- workloads ----------------------------------------------------------------------------------
def any_length_path(n):
    """The library's path for a length that is not a power of two (its planner's rule)."""
    m = n
    for f in (2, 3, 5, 7):
        while m % f == 0:
            m //= f
    if m == 1 and n <= 8192:
        return "mixed-radix path"
    if m == 1 and n <= 1 << 20 and any(n % d == 0 and n // d <= 8192
                                       for d in range(2, min(512, int(n ** 0.5)) + 1)):
        return "mixed-radix four-step path"
    return "chirp-z path"


class Workload:
    """Sizes, flop count and minimum traffic of one step."""

    def __init__(self, name):
        self.name = name
        self.pairing = False  # real rows: two rows per complex transform
        if name == "c2c_4096":
            self.kind, self.n, self.batch, self.dims, self.shift = "c2c_rt", 4096, 16384, 1, True
            self.desc = ("batched 1-D C2C fp32 N=4096 x 16384 rows, forward with fftshift as "
                         "(-1)^n premultiply then inverse")
        elif name == "c2c_1024":
            self.kind, self.n, self.batch, self.dims, self.shift = "c2c_fwd", 1024, 64, 1, False
            self.desc = "1-D C2C fp32 forward N=1024 x 64 rows"
        elif name.startswith("sweep_"):
            l = int(name.split("_")[1])
            self.kind, self.n, self.batch, self.dims, self.shift = "c2c_fwd", 1 << l, (1 << 26) >> l, 1, False
            self.desc = f"1-D C2C fp32 forward N=2^{l} x {(1 << 26) >> l} rows (3 tones + noise)"
        elif name.startswith("any_"):
            n = int(name.split("_")[1])
            self.kind, self.n, self.batch, self.dims, self.shift = "c2c_fwd", n, (1 << 26) // n, 1, False
            self.desc = (f"1-D C2C fp32 forward N={n} (not a power of two: {any_length_path(n)}) x "
                         f"{(1 << 26) // n} rows (3 tones + noise)")
        elif name.startswith("shift_"):
            n = int(name.split("_")[1])
            self.kind, self.n, self.batch, self.dims, self.shift = "shift", n, (1 << 26) // n, 1, True
            self.desc = (f"standalone fftshift by index rotation, {(1 << 26) // n} rows x {n} "
                         "complex64, out of place")
        elif name.startswith("realany_") or name.startswith("realanypair_"):
            n = int(name.split("_")[1])
            self.kind, self.n, self.batch, self.dims, self.shift = "real_rt", n, 2048, 1, False
            self.mmax = n // 3
            self.pairing = name.startswith("realanypair_")
            self.desc = (f"real rows 2048 x {n} (any length: {any_length_path(n)}), mmax={n // 3}: C2R "
                         "synthesis then R2C analysis, m-major spectrum" +
                         (", two rows per transform" if self.pairing else ""))
        elif name in ("real", "realpair"):
            self.kind, self.n, self.batch, self.dims, self.shift = "real_rt", 4096, 2048, 1, False
            self.mmax = 1365
            self.pairing = name == "realpair"
            self.desc = ("real rows 2048 x 4096, mmax=1365: C2R synthesis then R2C analysis, "
                         "m-major spectrum" + (", two rows per transform" if self.pairing else ""))
        elif name == "2d":
            self.kind, self.n, self.batch, self.dims, self.shift = "c2c_rt", 4096, 1, 2, True
            self.desc = ("2-D C2C fp32 4096x4096, forward with (-1)^(x+y) chessboard then "
                         "inverse")
        else:
            raise SystemExit(f"unknown workload {name}")
        n = self.n
        self.points = self.batch * (n * n if self.dims == 2 else n)
        self.log2n = math.log2(n)  # flop count 5*N*log2(N) for any N (CS598 metric)
        if self.kind == "shift":
            self.flops = 0.0
            self.min_bytes = 16 * self.batch * n  # one read + one write per point
        elif self.kind == "real_rt":
            m1 = self.mmax + 1
            self.flops = 2 * 2.5 * n * self.log2n * self.batch
            # synthesis reads the spectrum and writes reals; analysis the reverse
            self.min_bytes = 2 * (self.batch * m1 * 8 + self.batch * n * 4)
        else:
            per = 5.0 * n * self.log2n * (2 if self.dims == 2 else 1) * (n if self.dims == 2 else 1)
            ntr = 2 if self.kind == "c2c_rt" else 1
            self.flops = ntr * per * self.batch
            passes = 1 if (self.dims == 1 and n <= (1 << 14)) else 2  # one-pass, or two
            self.min_bytes = ntr * 16 * self.points  # one-pass minimum per transform
            self.pass_bytes = ntr * 16 * self.points * passes
        self.large = self.points * 8 > 2 * L2_BYTES

    @classmethod
    def with_rows(cls, name, rows):
        w = cls.__new__(cls)
        w.__dict__.update(cls(name).__dict__)
        scale = rows / w.batch
        w.batch = rows
        w.points = int(w.points * scale)
        w.flops *= scale
        w.min_bytes = int(w.min_bytes * scale)
        if hasattr(w, "pass_bytes"):
            w.pass_bytes = int(w.pass_bytes * scale)
        w.large = w.points * 8 > 2 * L2_BYTES
        w.desc += f" (rows overridden to {rows})"
        return w


def config_of(w, world):
    """The workload's `config` object (both arms print the same one)."""
    return {"workload": w.desc, "n": w.n, "batch_per_gpu": w.batch, "dims": w.dims,
            "l2": "inputs larger than L2" if w.large else "L2 flushed between steps",
            "parallelism": f"replicas x{world} (batch sharded, no collective)"}


def make_inputs(w, seed):
    from fft_signal_processing_gb300 import workloads as wl

    if w.kind == "real_rt":
        return wl.spectrum(seed, w.batch, w.mmax)
    if w.name == "c2c_4096":
        return wl.normal(seed, w.batch, w.n)
    if w.name == "c2c_1024":
        return wl.uniform(seed, w.batch, w.n)
    if w.name == "2d":
        return wl.image(seed, w.batch, w.n)
    return wl.tones(seed, w.batch, w.n)


# ---- clocks -------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return None
        under = [s for s in sm if mx and s > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(under), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- distributed helpers --------------------------------------------------------------------------
def dist_init(args):
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def job_rates(w, world, step_ms):
    """Whole-job GFLOP/s and minimum-traffic GB/s: every rank transforms its own batch of the
    workload (weak scaling), timed by the slowest rank's step."""
    return (w.flops * world / (step_ms * 1e-3) / 1e9, w.min_bytes * world / (step_ms * 1e-3) / 1e9)


def max_over_ranks(pg, v):
    if pg is None:
        return v
    import torch

    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def profile_traffic(kernel_key):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, if the
    kernel source has not changed since it was taken (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        data = json.load(open(path))
    except Exception:
        return None, None
    ent = data.get(kernel_key)
    if not ent or ent.get("source_sha") != kernel_source_sha(ent.get("source_files")):
        return None, None
    return ent.get("dram_bytes_per_launch"), ent.get("summary")


def kernel_source_sha(files=None):
    """Hash of the sources a kernel is built from (all of csrc/ when files is None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fft_signal_processing_gb300", "csrc")
    names = sorted(files) if files else sorted(
        f for f in os.listdir(csrc) if f.endswith((".cu", ".cuh", ".h")))
    for f in names:
        try:
            h.update(open(os.path.join(csrc, f), "rb").read())
        except OSError:
            return "missing:" + f
    return h.hexdigest()[:16]


# ---- CPU oracle timing (reference arm and cpu_baseline) -------------------------------------------
def oracle_step_sample(w, x, budget_s):
    """Time the fp64 oracle on a bounded sample of the workload; return (value, unit, cores,
    sample description, seconds)."""
    import numpy as np

    import oracle

    cores = oracle.num_threads()
    unit = "GFLOP/s"
    if w.kind == "shift":  # a rate in bytes moved (16 per point), like the GPU line
        per_row_flops = 16.0 * w.n

        def run(rows):
            oracle.fftshift_any(x[:rows], 1)
        unit_rows = w.batch
        unit = "GB/s"
    elif w.kind == "real_rt":
        per_row_flops = 2 * 2.5 * w.n * w.log2n

        pow2 = (w.n & (w.n - 1)) == 0

        def run(rows):  # the oracle's FFT path, or its direct sums for other lengths
            F = x[:rows]
            xr = oracle.c2r(F, w.n) if pow2 else oracle.c2r_direct(F, w.n)
            oracle.r2c(xr, w.mmax) if pow2 else oracle.r2c_direct(xr, w.mmax)
        unit_rows = w.batch
    elif w.dims == 2:
        per_row_flops = None

        def run(rows):  # rows = images
            img = x[:1]
            y = oracle.transform(img, -1, 2, w.shift)
            oracle.transform(y, +1, 2, w.shift)
        unit_rows = 1
    else:
        ntr = 2 if w.kind == "c2c_rt" else 1
        per_row_flops = ntr * 5.0 * w.n * w.log2n

        def run(rows):
            xs = x[:rows]
            y = oracle.transform(xs, -1, 1, w.shift)
            if ntr == 2:
                oracle.transform(y, +1, 1, w.shift)
        unit_rows = w.batch
    if w.dims == 2:
        t0 = time.perf_counter()
        run(1)
        dt = time.perf_counter() - t0
        gflops = w.flops / dt / 1e9
        return gflops, "GFLOP/s", cores, "one full 4096x4096 image, forward + inverse", dt
    rows = max(1, min(unit_rows, 8))
    while True:
        t0 = time.perf_counter()
        run(rows)
        dt = time.perf_counter() - t0
        if dt >= budget_s or rows >= unit_rows:
            break
        rows = min(unit_rows, max(rows * 2, int(rows * budget_s / max(dt, 1e-3) * 1.1)))
    gflops = per_row_flops * rows / dt / 1e9
    return gflops, unit, cores, f"{rows} of {unit_rows} rows of the same workload", dt


def run_reference(args, w):
    world, rank, local, pg = dist_init(args)
    if rank != 0:
        return
    x = make_inputs(w, 1)
    times = []
    sample = None
    for i in range(args.warmup + args.steps):
        v, unit, cores, sample, dt = oracle_step_sample(w, x, budget_s=max(1.0, 20.0 / max(1, args.steps + args.warmup)))
        if i >= args.warmup:
            times.append(v)
    value = statistics.median(times)
    metric = ("fftshift GB/s (16 B per complex point)" if w.kind == "shift"
              else "fp32 C2C FFT GFLOP/s (5N*log2N/t)")
    line = {
        "impl": "reference", "metric": metric, "value": value,
        "unit": unit, "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded)", "config": config_of(w, world),
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def host_link_ceiling(dev, nbytes=512 * 1024 * 1024, reps=3):
    """Plain pinned-memory copy rates on this machine (GB/s): host->device, device->host, and both
    at once on two streams (the ceiling of an end-to-end step that streams its input in and its
    result out).  Best of `reps`, CUDA events."""
    import torch

    hs = [torch.empty(nbytes, dtype=torch.uint8).pin_memory() for _ in range(2)]
    ds = [torch.empty(nbytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    s1, s2 = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def timed(fn):
        best = float("inf")
        for _ in range(reps):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(s1)
            s2.wait_event(e0)
            fn()
            e2 = torch.cuda.Event()
            e2.record(s2)
            s1.wait_event(e2)
            e1.record(s1)
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        return best

    def h2d():
        with torch.cuda.stream(s1):
            ds[0].copy_(hs[0], non_blocking=True)

    def d2h():
        with torch.cuda.stream(s1):
            hs[1].copy_(ds[1], non_blocking=True)

    def both():
        with torch.cuda.stream(s1):
            ds[0].copy_(hs[0], non_blocking=True)
        with torch.cuda.stream(s2):
            hs[1].copy_(ds[1], non_blocking=True)

    t_h2d, t_d2h, t_both = timed(h2d), timed(d2h), timed(both)
    del hs, ds
    return {"h2d_gbs": round(nbytes / (t_h2d * 1e-3) / 1e9, 1),
            "d2h_gbs": round(nbytes / (t_d2h * 1e-3) / 1e9, 1),
            "both_directions_gbs": round(2 * nbytes / (t_both * 1e-3) / 1e9, 1),
            "bytes_each_way": nbytes, "how": "pinned torch copy_, best of 3, CUDA events"}


# ---- the library arm --------------------------------------------------------------------------------
def main():
    args = parse()
    w = Workload(args.workload)
    if args.rows:
        w = Workload.with_rows(args.workload, args.rows)
    if args.impl == "reference":
        return run_reference(args, w)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")

    import numpy as np
    import torch

    world, rank, local, pg = dist_init(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import fft_signal_processing_gb300 as fx

    fx.lib()  # fail loudly if the CUDA library is missing
    stream = torch.cuda.Stream(device=dev)
    x_host = make_inputs(w, 1 + rank)

    with torch.cuda.stream(stream):
        if w.kind == "shift":
            xd = torch.from_numpy(x_host).to(dev)
            yd = torch.empty_like(xd)
            plans = []

            def launches():
                fx.shift_ptr(xd.data_ptr(), yd.data_ptr(), w.n, 1, w.batch, 1, False,
                             stream.cuda_stream)
                yield
        elif w.kind == "real_rt":
            syn = fx.Plan(w.n, w.batch, 1, fx.INVERSE, layout=fx.LAYOUT_REAL_MMAJOR, mmax=w.mmax,
                          pairing=w.pairing)
            ana = fx.Plan(w.n, w.batch, 1, fx.FORWARD, layout=fx.LAYOUT_REAL_MMAJOR, mmax=w.mmax,
                          pairing=w.pairing)
            F = torch.from_numpy(np.ascontiguousarray(x_host.T)).to(dev)  # m-major
            xr = torch.empty((w.batch, w.n), dtype=torch.float32, device=dev)
            G = torch.empty_like(F)
            plans = [syn, ana]

            def launches():
                syn.exec_c2r_ptr(F.data_ptr(), xr.data_ptr(), stream.cuda_stream)
                yield
                ana.exec_r2c_ptr(xr.data_ptr(), G.data_ptr(), stream.cuda_stream)
                yield
        else:
            fwd = fx.Plan(w.n, w.batch, w.dims, fx.FORWARD, shift=w.shift)
            inv = fx.Plan(w.n, w.batch, w.dims, fx.INVERSE, shift=w.shift) if w.kind == "c2c_rt" else None
            xd = torch.from_numpy(x_host).to(dev)
            yd = torch.empty_like(xd)
            zd = torch.empty_like(xd) if inv else None
            plans = [p for p in (fwd, inv) if p]

            def launches():
                fwd.exec_c2c_ptr(xd.data_ptr(), yd.data_ptr(), stream.cuda_stream)
                yield
                if inv:
                    inv.exec_c2c_ptr(yd.data_ptr(), zd.data_ptr(), stream.cuda_stream)
                    yield
        flush = None if w.large else torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    kernels_per_step = sum(1 for _ in launches())

    def kernels_of(plan):
        d = plan.describe()
        return int(d.split("kernels=")[1].split()[0])

    kper = sum(kernels_of(p) for p in plans) if plans else kernels_per_step

    def one_step(ev=None):
        if flush is not None:
            flush.zero_()
        if ev is not None:
            ev[0].record(stream)
        for i, _ in enumerate(launches()):
            if ev is not None:
                ev[i + 1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            one_step()
    torch.cuda.synchronize()

    # Timed region: windows of exactly K steps, each bracketed by a barrier and a device
    # synchronisation, with events around every launch on the launching stream.  The window is
    # repeated (the same count on every rank) until about --min-seconds have passed, so that the
    # clock sampler sees the kernels running; the step time is the median over windows.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(kernels_per_step + 1)]
           for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device() if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    clocks.start()
    time.sleep(0.3)

    def timed_window():
        barrier(pg)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for s in range(args.steps):
                one_step(evs[s])
        torch.cuda.synchronize()
        barrier(pg)
        wall = time.perf_counter() - t0
        return [[evs[s][i].elapsed_time(evs[s][i + 1]) for i in range(kernels_per_step)]
                for s in range(args.steps)], wall

    windows = [timed_window()]
    n_windows = int(min(200, max(3, math.ceil(args.min_seconds / max(windows[0][1], 1e-4)))))
    n_windows = int(max_over_ranks(pg, float(n_windows)))
    while len(windows) < n_windows:
        windows.append(timed_window())
    clk = clocks.stop()
    step_ms_windows = [statistics.mean(sum(pl) for pl in win) for win, _ in windows]
    step_ms_local = statistics.median(step_ms_windows)
    step_ms = max_over_ranks(pg, step_ms_local)
    launch_ms = [statistics.median(statistics.mean(pl[i] for pl in win) for win, _ in windows)
                 for i in range(kernels_per_step)]
    timed_seconds = sum(wall for _, wall in windows)

    gflops, gbs_min = job_rates(w, world, step_ms)

    # roofline of the dominant launch (one library call = one or two kernels)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or 6800.0
    dom = max(range(kernels_per_step), key=lambda i: launch_ms[i])
    if w.kind == "shift":
        dom_bytes, dom_kernels = w.min_bytes, 1
    elif w.kind == "real_rt":
        dom_bytes = (w.batch * (w.mmax + 1) * 8 + w.batch * w.n * 4)
        dom_kernels = 1
    else:
        dom_kernels = kernels_of(plans[min(dom, len(plans) - 1)])
        # read + write per kernel pass (four-step and 2-D: two full passes); the multi-pass
        # chirp-z call is rated against the one-pass minimum, 16 bytes per point
        multipass = "bluestein_multipass" in plans[min(dom, len(plans) - 1)].describe()
        dom_bytes = 16 * w.points * (1 if multipass else dom_kernels)
    achieved = dom_bytes / (launch_ms[dom] * 1e-3) / 1e9
    key = f"{w.name}:launch{dom}"
    traffic, _ = profile_traffic(key)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic,
                "peak_source": peak_src,
                "kernel": ("fft_shift" if not plans else
                           plans[min(dom, len(plans) - 1)].describe().split(" ")[0] +
                           (f" ({dom_kernels} kernels)" if dom_kernels > 1 else "")),
                "launch_ms": round(launch_ms[dom], 4),
                "algorithmic_bytes_per_launch": dom_bytes}

    # End to end through the C ABI with host buffers (pinned), copies inside the timed region.
    # The batch streams through in chunks of rows, as a user would feed it: per chunk one
    # host-to-device copy, the library's transforms, one device-to-host copy, on three streams
    # with two device buffers per stage, so copies of one chunk overlap compute of another.
    e2e = None
    if not args.no_e2e and w.kind not in ("real_rt", "shift") and w.dims == 1:
        nchunk = 8 if w.batch % 8 == 0 else 1
        rows_c = w.batch // nchunk
        xh = torch.from_numpy(x_host).pin_memory()
        outh = torch.empty_like(xh).pin_memory()
        fwd_c = fx.Plan(w.n, rows_c, 1, fx.FORWARD, shift=w.shift)
        inv_c = fx.Plan(w.n, rows_c, 1, fx.INVERSE, shift=w.shift) if inv else None
        bufs = [[torch.empty((rows_c, w.n), dtype=torch.complex64, device=dev) for _ in range(3)]
                for _ in range(2)]
        s_in, s_cmp, s_out = (torch.cuda.Stream(device=dev) for _ in range(3))
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_cmp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        for e in ev_cmp + ev_out:
            e.record(s_cmp)

        def e2e_step():
            for c in range(nchunk):
                b = c % 2
                xb, yb, zb = bufs[b]
                lo, hi = c * rows_c, (c + 1) * rows_c
                s_in.wait_event(ev_cmp[b])  # xb free
                with torch.cuda.stream(s_in):
                    xb.copy_(xh[lo:hi], non_blocking=True)
                ev_in[b].record(s_in)
                s_cmp.wait_event(ev_in[b])
                s_cmp.wait_event(ev_out[b])  # zb free
                fwd_c.exec_c2c_ptr(xb.data_ptr(), yb.data_ptr(), s_cmp.cuda_stream)
                res_b = yb
                if inv_c is not None:
                    inv_c.exec_c2c_ptr(yb.data_ptr(), zb.data_ptr(), s_cmp.cuda_stream)
                    res_b = zb
                ev_cmp[b].record(s_cmp)
                s_out.wait_event(ev_cmp[b])
                with torch.cuda.stream(s_out):
                    outh[lo:hi].copy_(res_b, non_blocking=True)
                ev_out[b].record(s_out)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        barrier(pg)
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(s_in)
        for _ in range(args.steps):
            e2e_step()
        ev1.record(s_out)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(pg, ev0.elapsed_time(ev1) / args.steps)
        link_gbs = round(2 * xh.numel() * xh.element_size() / (e2e_ms * 1e-3) / 1e9, 1)
        link = host_link_ceiling(dev)
        e2e = {"value": round(w.flops * world / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GFLOP/s",
               "h2d_bytes_per_step": int(xh.numel() * xh.element_size()),
               "d2h_bytes_per_step": int(outh.numel() * outh.element_size()),
               "ms_per_step": round(e2e_ms, 4), "chunks_per_step": nchunk,
               "h2d_d2h_gbs": link_gbs, "host_link": link,
               "host_link_frac": round(link_gbs / link["both_directions_gbs"], 3)}
        fwd_c.close()
        if inv_c is not None:
            inv_c.close()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        v, unit, cores, sample, dt = oracle_step_sample(w, x_host, budget_s=10.0)
        cpu = {"value": round(v, 3), "unit": unit, "cores": cores, "kind": "oracle",
               "sample": sample, "seconds": round(dt, 2)}

    if rank == 0:
        metric, value, unit = "fp32 C2C FFT GFLOP/s (5N*log2N/t)", round(gflops, 1), "GFLOP/s"
        if w.kind == "shift":  # pure data movement: the rate is bytes, not flops
            metric, value, unit = "fftshift GB/s (16 B per complex point)", round(gbs_min, 1), "GB/s"
        line = {
            "metric": metric,
            "value": value, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded numpy generators)",
            "config": config_of(w, world),
            "hbm_gbs_min_traffic": round(gbs_min, 1),
            "hbm_frac_min_traffic": round(gbs_min / world / peak, 4),
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": kper * args.steps * len(windows),
            "timed_windows": {"count": len(windows), "steps_each": args.steps,
                              "seconds": round(timed_seconds, 3),
                              "ms_per_step_min": round(min(step_ms_windows), 4),
                              "ms_per_step_max": round(max(step_ms_windows), 4)},
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    for p in plans:
        p.close()
    if pg is not None:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
