"""Build libdflash.so in-tree with nvcc for sm_103a (one -gencode), compiling
the translation units in parallel and linking against the shared CUDA
runtime so the library shares torch's runtime in-process."""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libdflash.so")
# The checked variant: device bounds assertions (DFLASH_CHECKED) that report
# through the status word instead of trapping.
LIB_CHECKED = os.path.join(OUT_DIR, "libdflash_checked.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         f"-I{INCLUDE}"]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(src: str, verbose: bool, checked: bool = False) -> str:
    obj = os.path.join(OUT_DIR, os.path.basename(src) + (".checked.o" if checked else ".o"))
    cmd = [NVCC, *ARCH, *FLAGS, *(["-DDFLASH_CHECKED"] if checked else []), "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
    if verbose and r.stderr:
        print(r.stderr)
    return obj


def _link(objs, lib: str) -> None:
    tmp = lib + f".{os.getpid()}.tmp"
    cmd = [NVCC, *ARCH, "-shared", "-cudart", "shared", "-Xlinker", "-rpath,/usr/local/cuda/lib64",
           "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every .cu under csrc/ twice (the normal and the checked
    variant, all in parallel) and link libdflash.so and
    libdflash_checked.so; returns the normal library's path."""
    if not force and up_to_date(LIB) and up_to_date(LIB_CHECKED):
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    srcs = _sources()
    jobs = [(src, False) for src in srcs] + [(src, True) for src in srcs]
    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda j: _compile(j[0], verbose, j[1]), jobs))
    _link(objs[:len(srcs)], LIB)
    _link(objs[len(srcs):], LIB_CHECKED)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
