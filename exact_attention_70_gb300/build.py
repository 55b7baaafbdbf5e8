"""Build ``libattn.so`` in-tree with nvcc for sm_103a (translation units compiled in parallel).

Static CUDA runtime; the driver's tensor-map encoder is reached through the runtime's
driver-entry-point query, so the library loads on a machine without a GPU driver.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libattn.so")
# The debugging build with device bounds checks (-DATTN_CHECK_BOUNDS): a separate library.
BUILD_CHECKED = os.path.join(HERE, "_build_checked")
LIB_CHECKED = os.path.join(BUILD_CHECKED, "libattn.so")
SOURCES = ["attn_api.cu", "fwd_kernel.cu", "decode_kernel.cu", "decode_noalloc.cu", "selftest.cu", "kvcache.cu", "bwd_kernel.cu", "fwd_fp8_kernel.cu", "quantize_fp8.cu"]
HEADERS = ["ptx.cuh", "kernels.h", "tile_math.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def _flags(extra=()):
    return [NVCC, *ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
            f"-I{os.path.join(ROOT, 'include')}", *extra]


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          check_bounds: bool = False) -> str:
    """Compile libattn.so (or, with check_bounds, the debugging library whose kernels check
    their stores and TMA coordinates and report violations in the status word)."""
    build_dir, lib = (BUILD_CHECKED, LIB_CHECKED) if check_bounds else (BUILD, LIB)
    extra = ["-DATTN_CHECK_BOUNDS"] if check_bounds else []
    os.makedirs(build_dir, exist_ok=True)
    deps = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "attn.h")]
    dep_time = max(os.path.getmtime(d) for d in deps)
    procs, objs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or not os.path.exists(o) or os.path.getmtime(o) < max(dep_time, os.path.getmtime(s)):
            cmd = _flags(extra + (["-Xptxas", "-v"] if ptxas_info else [])) + ["-c", s, "-o",
                                                                               o + ".tmp"]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT), o, s))
    failed = []
    for p, o, s in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append(f"{s}:\n{text}")
        else:
            os.replace(o + ".tmp", o)
            if verbose or ptxas_info:
                print(text, file=sys.stderr)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs):
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.check_call([NVCC, *ARCH, "-shared", "-o", tmp, *objs, "-ldl"])
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                check_bounds="--check-bounds" in sys.argv))
