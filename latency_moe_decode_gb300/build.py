"""Build the engine's shared library (libdec.so) in-tree with nvcc for sm_103a."""
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libdec.so")
SOURCES = ["dec_engine.cu", "dec_wide.cu"]
HEADERS = ["dec_common.h", "dec_prims.cuh", "dec_kernel.cuh", "dec_wide.cuh", "dec_wide_host.h"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "dec.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    tag = f".tmp{os.getpid()}"
    tmp = LIB + tag
    flags = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
             "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    if verbose:
        flags.insert(0, "-Xptxas=-v")
    if os.environ.get("DEC_DIAG") == "1":  # diagnostics build: event trace and per-CTA stamps
        flags += ["-DDEC_TRACE=1", "-DDEC_STAMPS=1"]
    # one object per translation unit, compiled in parallel, then linked
    objs = [os.path.join(PKG, os.path.splitext(s)[0] + tag + ".o") for s in SOURCES]
    procs = [subprocess.Popen([nvcc()] + flags + ["-c", "-o", o, os.path.join(CSRC, s)])
             for s, o in zip(SOURCES, objs)]
    rcs = [pr.wait() for pr in procs]
    try:
        if any(rcs):
            raise subprocess.CalledProcessError(max(rcs), "nvcc -c")
        subprocess.run([nvcc(), "-shared", "-o", tmp] + objs, check=True)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
