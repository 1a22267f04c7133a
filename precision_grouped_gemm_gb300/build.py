"""Build libpgg.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each .cu translation unit compiles in parallel to an object under _build/, then
nvcc links them into precision_grouped_gemm_gb300/libpgg.so with the CUDA
runtime linked statically (the library then loads on machines without a GPU
driver, which the CPU-side ABI tests rely on).  The driver API entry point the
library needs (tensor-map encoding) is fetched at run time.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libpgg.so")
SOURCES = ["pgg_api.cu", "gemm_bf16.cu", "mx_quant.cu", "gemm_mx.cu", "moe_glue.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(verbose: bool = False, force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(ROOT, "include", "pgg.h"))
    cc = nvcc()

    def compile_one(src):
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        if not force and _newer(o, [s] + headers):
            return o
        cmd = [cc, *ARCH, *FLAGS, "-Xptxas", "-v", "-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        with open(o + ".log", "w") as f:
            f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr[-4000:]}")
        if verbose:
            print(r.stderr)
        return o

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or not _newer(LIB, objs):
        cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", LIB, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))


# Kernel families with DRAM counters in profiles/traffic.json, and the sources each one's
# kernels cannot depend on (separate translation units): a family's counters stay valid
# while the sources it is built from are unchanged.
DIGEST_EXCLUDE = {
    "bf16": ("gemm_mx.cu", "mx_quant.cu", "moe_glue.cu"),    # BF16 grouped GEMM family
    "mx": ("gemm_bf16.cu", "gemm_bf16.cuh", "moe_glue.cu"),  # block-scaled GEMM + MX quantizers
}


def source_digest(family: str) -> str:
    """sha256 over the CUDA sources and headers a kernel family is built from (identifies the
    kernels a profile was taken on)."""
    import hashlib
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cuh", ".h")) and name not in DIGEST_EXCLUDE[family]:
            with open(os.path.join(CSRC, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]
