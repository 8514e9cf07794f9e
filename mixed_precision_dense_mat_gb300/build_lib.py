"""Build libcr.so in-tree with nvcc for sm_103a (one -gencode, translation units compiled in
parallel).  Used by __graft_entry__.build() and by the package loader."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "libcr.so")
SOURCES = ["api.cu", "cov.cu", "policy.cu", "fp64.cu", "diag.cu", "tc.cu", "chol.cu", "sim.cu", "calib.cu", "krige.cu", "peaks.cu",
           "ozaki.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=default",
         "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, obj: str) -> tuple[str, str]:
    cmd = [nvcc(), *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{p.stdout}\n{p.stderr}")
    return src, p.stderr


def build(verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    objs = [os.path.join(OUT_DIR, s.replace(".cu", ".o")) for s in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        logs = list(ex.map(lambda a: _compile(*a), zip(SOURCES, objs)))
    if verbose:
        for src, log in logs:
            sys.stderr.write(f"--- {src}\n{log}")
    # cuBLAS (the Ozaki product's FP16 slice GEMMs) from the toolkit next to nvcc
    libdir = os.path.realpath(os.path.join(os.path.dirname(nvcc()), "..", "lib64"))
    cmd = [nvcc(), *ARCH, "-shared", "-o", LIB, *objs, "-lcudart_static", "-L" + libdir, "-lcublas",
           "-Xlinker", "-rpath=" + libdir, "-lrt", "-ldl", "-lpthread"]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
    with open(os.path.join(OUT_DIR, "ptxas.log"), "w") as f:
        for src, log in logs:
            f.write(f"--- {src}\n{log}")
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
