"""Build libgbfft.so (the CUDA kernels and the C ABI) in-tree with nvcc for sm_103a.

Each translation unit under csrc/ is compiled in parallel to an object file, then linked into
fft_signal_processing_gb300/libgbfft.so.  Objects are rebuilt only when a source or header is
newer than them.  build(checked=True) makes the checked variant libgbfft_checked.so from the
same sources with -DGBFFT_CHECKED (device-side index checks that report FFT_ERR_BOUNDS), in an
object directory of its own; tests load it through GBFFT_CHECKED=1.
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgbfft.so")
OBJ_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libgbfft_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgbfft.so")


def _deps():
    hdrs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
    hdrs.append(os.path.join(ROOT, "include", "gbfft.h"))
    return max(os.path.getmtime(h) for h in hdrs)


def _compile(src: str, extra, verbose: bool, objdir: str = OBJ) -> str:
    obj = os.path.join(objdir, os.path.basename(src) + ".o")
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), _deps()):
        return obj
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + list(extra) + ["-c", src, "-o", obj + ".tmp"]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if verbose:
        sys.stderr.write(r.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False, verbose: bool = False, extra=(), checked: bool = False) -> str:
    objdir, lib = (OBJ_CHECKED, LIB_CHECKED) if checked else (OBJ, LIB)
    extra = list(extra) + (["-DGBFFT_CHECKED"] if checked else [])
    os.makedirs(objdir, exist_ok=True)
    if force:
        for o in glob.glob(os.path.join(objdir, "*.o")):
            os.remove(o)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    workers = max(1, min(len(srcs), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, verbose, objdir), srcs))
    if (not force and os.path.exists(lib)
            and os.path.getmtime(lib) >= max(os.path.getmtime(o) for o in objs)):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link of {os.path.basename(lib)} failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                checked="--checked" in sys.argv))
