"""Build libmotion_gb300.so in-tree with nvcc for sm_103a (one -gencode, the
translation units compiled in parallel, then linked into one shared object).

``build(checked=True)`` builds the bounds-checked variant,
libmotion_gb300_checked.so (MG_BOUNDS_CHECK=1: every shared- and global-memory
access of the motion kernels is checked against its buffer, a failed check
skips the access and sets bit 1 of the device error word); the tests run it
on small cases, as the stand-in for a memory checker."""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
LIB_NAME = "libmotion_gb300.so"
CHECKED_LIB_NAME = "libmotion_gb300_checked.so"
# the instruction-throughput microbenchmark behind the integer co-bound
# (pipe_rates.cu; a library of its own, not part of the motion library)
PIPE_LIB_NAME = "libpipe_rates_gb300.so"
PIPE_SOURCE = "pipe_rates.cu"
SOURCES = ["motion_capi.cu", "motion_tile.cu", "motion_tma.cu", "psnr_sse.cu", "motion_noalloc.cu",
           "moment.cu", "repitch.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def lib_path(checked: bool = False) -> str:
    return os.path.join(OUT_DIR, CHECKED_LIB_NAME if checked else LIB_NAME)


def pipe_lib_path() -> str:
    return os.path.join(OUT_DIR, PIPE_LIB_NAME)


def build_pipe_rates(force: bool = False) -> str:
    """Build libpipe_rates_gb300.so (one translation unit)."""
    src = os.path.join(CSRC, PIPE_SOURCE)
    out = pipe_lib_path()
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(OUT_DIR, exist_ok=True)
    cmd = [nvcc()] + ARCH + ["-O3", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden", "-shared",
                             "-o", out + ".tmp", src]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {PIPE_SOURCE}:\n{r.stdout}\n{r.stderr}")
    os.replace(out + ".tmp", out)
    return out


def _newest_source_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f != PIPE_SOURCE]
    files.append(os.path.join(INCLUDE, "motion.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def up_to_date(checked: bool = False) -> bool:
    p = lib_path(checked)
    return os.path.exists(p) and os.path.getmtime(p) >= _newest_source_mtime()


def build(force: bool = False, verbose: bool = False, extra_flags: tuple[str, ...] = (),
          checked: bool = False) -> str:
    if not force and up_to_date(checked):
        return lib_path(checked)
    os.makedirs(OUT_DIR, exist_ok=True)
    obj_dir = os.path.join(OUT_DIR, "obj_checked" if checked else "obj")
    if checked:
        extra_flags = tuple(extra_flags) + ("-DMG_BOUNDS_CHECK=1",)
    os.makedirs(obj_dir, exist_ok=True)
    cc = nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                     "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"] + list(extra_flags)
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src: str) -> str:
        obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path(checked) + ".tmp"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs + ["-Xcompiler", "-fPIC"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path(checked))
    return lib_path(checked)


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
