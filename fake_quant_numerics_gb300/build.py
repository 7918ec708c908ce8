"""Build of the CUDA library libqat.so (nvcc, sm_103a), in-tree.

Each translation unit is compiled in its own nvcc process (in parallel), then
linked into ``fake_quant_numerics_gb300/libqat.so``.  Floating-point flags pin
IEEE behaviour: no FMA contraction, IEEE division and square root, no
flush-to-zero.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libqat.so")

SOURCES = ["qat_abi.cu", "kernels_tensor.cu", "kernels_fused.cu", "kernels_fp8.cu",
           "kernels_misc.cu", "kernels_optim.cu", "kernels_cols.cu", "kernels_pct.cu", "kernels_block.cu", "kernels_onchip.cu",
           "kernels_unaligned.cu", "qat_noalloc.cu"]
# sources compiled a second time with QAT_SR=1: their stochastic-rounding
# kernels and *_sr launchers (object <name>_sr.o)
SR_SOURCES = ["kernels_tensor.cu", "kernels_fused.cu", "kernels_fp8.cu", "kernels_cols.cu"]
HEADERS = ["qat_device.cuh", "qat_launch.h", "qat_sr.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-fmad=false",
           "-prec-div=true", "-prec-sqrt=true", "-ftz=false", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return "nvcc"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, extra_flags=()) -> str:
    """Compile stale translation units and (re)link libqat.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "qat.h")]
    jobs, objs = [], []
    units = [(src, src.replace(".cu", ".o"), []) for src in SOURCES]
    units += [(src, src.replace(".cu", "_sr.o"), ["-DQAT_SR=1"]) for src in SR_SOURCES]
    # the longest translation units first, so the parallel build ends sooner
    units.sort(key=lambda u: u[0] != "kernels_fused.cu")
    for src, oname, defs in units:
        sp = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, oname)
        objs.append(obj)
        if verbose or _stale(obj, [sp, *hdrs, __file__]):
            cmd = [nvcc, *ARCH, *NVFLAGS, *defs, *extra_flags, "-c", sp, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stderr

    if jobs:
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
            for out in ex.map(run, jobs):
                if verbose and out:
                    print(out)
    if jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        r = subprocess.run([nvcc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True,
                           text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys

    print(build(verbose="-v" in sys.argv))
