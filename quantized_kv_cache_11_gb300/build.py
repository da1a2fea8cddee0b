"""Build libkvq.so (the C-ABI library) in-tree with nvcc for sm_103a.

    python -m quantized_kv_cache_11_gb300.build [--verbose]

Each .cu translation unit compiles in parallel to an object file, then nvcc
links them into ``quantized_kv_cache_11_gb300/libkvq.so``.  No CMake.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libkvq.so")
SOURCES = ["kvq_api.cu", "kvq_quantize.cu", "kvq_decode.cu", "kvq_trizone_build.cu",
           "kvq_trizone_decode.cu", "kvq_rdkv.cu", "kvq_decode_rope.cu", "kvq_selftest.cu",
           "kvq_decode_cps2.cu", "kvq_decode_cps4.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# IEEE-exact fp32 division and no flush-to-zero: the quantizer must match the
# oracle bit for bit.  Never --use_fast_math.
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-prec-div=true",
         "-prec-sqrt=true", "-ftz=false", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources_newer(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    for f in os.listdir(CSRC):
        if os.path.getmtime(os.path.join(CSRC, f)) > t:
            return True
    inc = os.path.join(os.path.dirname(HERE), "include")
    if any(os.path.getmtime(os.path.join(inc, f)) > t for f in os.listdir(inc)):
        return True
    return os.path.getmtime(__file__) > t


def build(force: bool = False, verbose: bool = False, extra: list | None = None) -> str:
    """Compile and link; returns the library path.  Skips work when up to date."""
    if not force and not _sources_newer(LIB):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = list(extra or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose="--verbose" in sys.argv))
