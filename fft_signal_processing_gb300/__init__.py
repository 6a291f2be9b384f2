"""Batched fp32 FFT for one GB300 GPU: Python binding of libgbfft.so (include/gbfft.h).

The binding only marshals arguments: it checks dtypes, shapes and devices of torch tensors
and passes raw device pointers and the current CUDA stream to the C ABI.  Every step of a
transform runs in the library's CUDA kernels; if the library is missing or fails to load, the
calls raise instead of computing anything another way.

    from fft_signal_processing_gb300 import Plan, FORWARD, INVERSE
    p = Plan(4096, batch=16384, direction=FORWARD, shift=True)
    y = p.c2c(x)                # x: complex64 CUDA tensor [16384, 4096]
    Plan(1000, 64).c2c(z)                                   # any length up to 2^20
    Plan(4096, 2048, layout=LAYOUT_REAL_MMAJOR, mmax=1365).r2c(rows)   # band-limited real rows
    Plan(1024, 1, dims=2, ny=512, direction=INVERSE, normalize=True).c2c(img)  # 512 x 1024
    shift(y)                                                # standalone fftshift
"""
import ctypes
import os

FORWARD = -1
INVERSE = +1
LAYOUT_C2C = 0
LAYOUT_REAL_ROWMAJOR = 1
LAYOUT_REAL_MMAJOR = 2

FFT_OK = 0
FFT_ERR_INVALID_ARG = -1
FFT_ERR_UNSUPPORTED_SIZE = -2
FFT_ERR_MISALIGNED = -3
FFT_ERR_OOM = -4
FFT_ERR_CUDA = -5
FFT_ERR_TIMEOUT = -6
FFT_ERR_BOUNDS = -7

# GBFFT_CHECKED=1 in the environment (tests) loads the checked build, libgbfft_checked.so:
# the same kernels with device-side index checks that report FFT_ERR_BOUNDS.
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "libgbfft_checked.so" if os.environ.get("GBFFT_CHECKED") == "1"
                        else "libgbfft.so")

# Exported C symbols (kept in step with include/gbfft.h; checked by the tests).
ABI_SYMBOLS = (
    "fft_plan_create", "fft_plan_set_band_limit", "fft_plan_workspace_bytes",
    "fft_plan_describe", "fft_plan_query", "fft_exec_c2c", "fft_exec_r2c", "fft_exec_c2r",
    "fft_plan_check", "fft_plan_destroy", "fft_status_string", "fft_version",
    "fft_exec_c2c_noalloc", "fft_plan_set_wait_timeout", "fft_shift", "fft_plan_create_2d",
    "fft_plan_query_2d", "fft_plan_set_normalization", "fft_plan_set_real_pairing",
    "fft_plan_set_diagnostic",
)

_LIB = None


class GbfftError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = int(status)
        msg = status_string(status)
        super().__init__(f"{what}: {msg}" if what else msg)


def lib():
    """Load libgbfft.so (built in-tree by __graft_entry__.build()); raise if unavailable."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{os.path.basename(LIB_PATH)} is not built ({LIB_PATH}); "
                               "run `python -c 'import __graft_entry__ as g; g.build()'` "
                               "(or `python fft_signal_processing_gb300/_build.py --checked`)")
        L = ctypes.CDLL(LIB_PATH)
        i64, ci, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
        L.fft_plan_create.argtypes = [i64, i64, ci, ci, ci, ci, ctypes.POINTER(vp)]
        L.fft_plan_set_band_limit.argtypes = [vp, i64]
        L.fft_plan_set_normalization.argtypes = [vp, ci]
        L.fft_plan_set_real_pairing.argtypes = [vp, ci]
        L.fft_plan_set_diagnostic.argtypes = [vp, ci]
        L.fft_plan_workspace_bytes.argtypes = [vp, ctypes.POINTER(sz)]
        L.fft_plan_describe.argtypes = [vp, ctypes.c_char_p, sz]
        L.fft_plan_query.argtypes = [i64, i64, ci, ci, ci, ci, ctypes.c_char_p, sz]
        L.fft_plan_create_2d.argtypes = [i64, i64, i64, ci, ci, ctypes.POINTER(vp)]
        L.fft_plan_query_2d.argtypes = [i64, i64, i64, ci, ci, ctypes.c_char_p, sz]
        L.fft_exec_c2c.argtypes = [vp, vp, vp, vp]
        L.fft_shift.argtypes = [vp, vp, i64, i64, i64, ci, ci, vp]
        L.fft_exec_r2c.argtypes = [vp, vp, vp, vp]
        L.fft_exec_c2r.argtypes = [vp, vp, vp, vp]
        L.fft_plan_check.argtypes = [vp]
        L.fft_plan_destroy.argtypes = [vp]
        L.fft_status_string.argtypes = [ci]
        L.fft_status_string.restype = ctypes.c_char_p
        L.fft_version.argtypes = []
        L.fft_exec_c2c_noalloc.argtypes = [i64, i64, ci, ci, vp, vp, vp]
        L.fft_plan_set_wait_timeout.argtypes = [vp, ctypes.c_uint64]
        for name in ABI_SYMBOLS:
            if name != "fft_status_string":
                getattr(L, name).restype = ci
        _LIB = L
    return _LIB


def status_string(status) -> str:
    return lib().fft_status_string(int(status)).decode()


def _check(rc, what):
    if rc != FFT_OK:
        raise GbfftError(rc, what)


def query(n, batch, dims=1, direction=FORWARD, layout=LAYOUT_C2C, shift=False, ny=None) -> str:
    """Host-only: the execution path a plan with these parameters would use."""
    buf = ctypes.create_string_buffer(1024)
    if dims == 2 and ny is not None and int(ny) != int(n):
        _check(lib().fft_plan_query_2d(int(n), int(ny), int(batch), int(direction),
                                       int(bool(shift)), buf, len(buf)), "fft_plan_query_2d")
        return buf.value.decode()
    _check(lib().fft_plan_query(int(n), int(batch), int(dims), int(direction), int(layout),
                                int(bool(shift)), buf, len(buf)), "fft_plan_query")
    return buf.value.decode()


def shift_ptr(in_ptr, out_ptr, nx, ny=1, batch=1, dims=1, inverse=False, stream_ptr=0):
    """fftshift (or ifftshift) of raw device buffers by index rotation (fft_shift)."""
    _check(lib().fft_shift(ctypes.c_void_p(in_ptr), ctypes.c_void_p(out_ptr), int(nx), int(ny),
                           int(batch), int(dims), int(bool(inverse)), ctypes.c_void_p(stream_ptr)),
           "fft_shift")


def shift(x, dims=1, inverse=False, out=None, stream=None):
    """fftshift / ifftshift of a complex64 CUDA tensor: the last axis (dims=1) or the last two
    axes (dims=2) of every row or image rotate by half their extent (rounded down); out=x runs
    in place (even extents only)."""
    import torch

    if x.dtype != torch.complex64 or not x.is_cuda or not x.is_contiguous():
        raise TypeError("shift: expected a contiguous complex64 CUDA tensor")
    nx = x.shape[-1]
    ny = x.shape[-2] if dims == 2 else 1
    if out is None:
        out = torch.empty_like(x)
    elif out.dtype != torch.complex64 or out.shape != x.shape or not out.is_contiguous():
        raise TypeError("shift: out must match x")
    shift_ptr(x.data_ptr(), out.data_ptr(), nx, ny, x.numel() // (nx * ny), dims, inverse,
              _stream_ptr(stream).value or 0)
    return out


def exec_c2c_noalloc(n, batch, direction, shift, in_ptr, out_ptr, stream_ptr=0):
    """Allocation-free batched C2C transform on raw device pointers (fft_exec_c2c_noalloc)."""
    _check(lib().fft_exec_c2c_noalloc(int(n), int(batch), int(direction), int(bool(shift)),
                                      ctypes.c_void_p(in_ptr), ctypes.c_void_p(out_ptr),
                                      ctypes.c_void_p(stream_ptr)), "fft_exec_c2c_noalloc")


def _stream_ptr(stream):
    import torch

    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(int(s.cuda_stream))


class Plan:
    """A planned batched transform on the current CUDA device (see include/gbfft.h).

    dims=1: rows of n points; dims=2: ny x n images (ny = n unless given; both powers of two
    up to 4096, rows of n points then columns of ny points).  direction: FORWARD / INVERSE,
    unnormalised.  layout: LAYOUT_C2C, or LAYOUT_REAL_ROWMAJOR / LAYOUT_REAL_MMAJOR for the
    band-limited real-row analysis (FORWARD, r2c) / synthesis (INVERSE, c2r) with mmax.
    shift: fftshift folded in as the (-1)^j chessboard (C2C only).  pairing: real layouts only,
    two real rows per complex transform (fft_plan_set_real_pairing).
    """

    def __init__(self, n, batch=1, dims=1, direction=FORWARD, layout=LAYOUT_C2C, shift=False,
                 mmax=None, ny=None, normalize=False, pairing=False):
        self.n, self.batch, self.dims = int(n), int(batch), int(dims)
        self.direction, self.layout, self.shift = int(direction), int(layout), bool(shift)
        self.ny = (self.n if ny is None else int(ny)) if self.dims == 2 else 1
        h = ctypes.c_void_p()
        if self.dims == 2 and self.ny != self.n:
            _check(lib().fft_plan_create_2d(self.n, self.ny, self.batch, self.direction,
                                            int(self.shift), ctypes.byref(h)), "fft_plan_create_2d")
        else:
            _check(lib().fft_plan_create(self.n, self.batch, self.dims, self.direction,
                                         self.layout, int(self.shift), ctypes.byref(h)),
                   "fft_plan_create")
        self._h = h
        self.mmax = None
        if normalize:
            self.set_normalization(True)
        if layout != LAYOUT_C2C:
            self.mmax = (self.n - 1) // 2 if mmax is None else int(mmax)
            _check(lib().fft_plan_set_band_limit(self._h, self.mmax), "fft_plan_set_band_limit")
        if pairing:
            _check(lib().fft_plan_set_real_pairing(self._h, 1), "fft_plan_set_real_pairing")

    @property
    def handle(self):
        return self._h

    def describe(self) -> str:
        buf = ctypes.create_string_buffer(1024)
        _check(lib().fft_plan_describe(self._h, buf, len(buf)), "fft_plan_describe")
        return buf.value.decode()

    def workspace_bytes(self) -> int:
        b = ctypes.c_size_t()
        _check(lib().fft_plan_workspace_bytes(self._h, ctypes.byref(b)), "workspace_bytes")
        return int(b.value)

    def check(self):
        _check(lib().fft_plan_check(self._h), "fft_plan_check")

    def set_normalization(self, on: bool = True):
        """Scale the output by 1/n (1/(nx*ny) for 2-D), or not (the default)."""
        _check(lib().fft_plan_set_normalization(self._h, int(bool(on))),
               "fft_plan_set_normalization")

    def set_index_only(self, on: bool = True):
        """Test hook: the kernels move values through their load/store epilogues only
        (fft_plan_set_diagnostic with FFT_DIAG_INDEX_ONLY)."""
        _check(lib().fft_plan_set_diagnostic(self._h, 1 if on else 0), "fft_plan_set_diagnostic")

    def set_wait_timeout(self, ns: int):
        """Limit of every device-side wait of this plan's kernels (0: give up at once)."""
        _check(lib().fft_plan_set_wait_timeout(self._h, int(ns)), "fft_plan_set_wait_timeout")

    def close(self):
        if getattr(self, "_h", None):
            lib().fft_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- shapes ----
    def complex_shape(self):
        return (self.batch, self.n) if self.dims == 1 else (self.batch, self.ny, self.n)

    def spectrum_shape(self):
        m1 = self.mmax + 1
        return (m1, self.batch) if self.layout == LAYOUT_REAL_MMAJOR else (self.batch, m1)

    def real_shape(self):
        return (self.batch, self.n)

    # ---- raw-pointer execution (device pointers as ints) ----
    def exec_c2c_ptr(self, in_ptr, out_ptr, stream_ptr=0):
        _check(lib().fft_exec_c2c(self._h, ctypes.c_void_p(in_ptr), ctypes.c_void_p(out_ptr),
                                  ctypes.c_void_p(stream_ptr)), "fft_exec_c2c")

    def exec_r2c_ptr(self, in_ptr, out_ptr, stream_ptr=0):
        _check(lib().fft_exec_r2c(self._h, ctypes.c_void_p(in_ptr), ctypes.c_void_p(out_ptr),
                                  ctypes.c_void_p(stream_ptr)), "fft_exec_r2c")

    def exec_c2r_ptr(self, in_ptr, out_ptr, stream_ptr=0):
        _check(lib().fft_exec_c2r(self._h, ctypes.c_void_p(in_ptr), ctypes.c_void_p(out_ptr),
                                  ctypes.c_void_p(stream_ptr)), "fft_exec_c2r")

    # ---- torch-tensor execution ----
    @staticmethod
    def _need(t, dtype, numel, what):
        import torch

        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{what}: expected a CUDA tensor")
        if t.dtype != dtype:
            raise TypeError(f"{what}: expected {dtype}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{what}: tensor must be contiguous")
        if t.numel() != numel:
            raise ValueError(f"{what}: expected {numel} elements, got {t.numel()}")

    def c2c(self, x, out=None, stream=None):
        import torch

        numel = self.batch * self.n * self.ny
        self._need(x, torch.complex64, numel, "c2c input")
        if out is None:
            out = torch.empty(self.complex_shape(), dtype=torch.complex64, device=x.device)
        self._need(out, torch.complex64, numel, "c2c output")
        _check(lib().fft_exec_c2c(self._h, ctypes.c_void_p(x.data_ptr()),
                                  ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream)),
               "fft_exec_c2c")
        return out

    def r2c(self, x, out=None, stream=None):
        import torch

        self._need(x, torch.float32, self.batch * self.n, "r2c input")
        if out is None:
            out = torch.empty(self.spectrum_shape(), dtype=torch.complex64, device=x.device)
        self._need(out, torch.complex64, self.batch * (self.mmax + 1), "r2c output")
        _check(lib().fft_exec_r2c(self._h, ctypes.c_void_p(x.data_ptr()),
                                  ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream)),
               "fft_exec_r2c")
        return out

    def c2r(self, F, out=None, stream=None):
        import torch

        self._need(F, torch.complex64, self.batch * (self.mmax + 1), "c2r input")
        if out is None:
            out = torch.empty(self.real_shape(), dtype=torch.float32, device=F.device)
        self._need(out, torch.float32, self.batch * self.n, "c2r output")
        _check(lib().fft_exec_c2r(self._h, ctypes.c_void_p(F.data_ptr()),
                                  ctypes.c_void_p(out.data_ptr()), _stream_ptr(stream)),
               "fft_exec_c2r")
        return out
