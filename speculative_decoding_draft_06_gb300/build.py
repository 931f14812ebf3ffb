"""Compile the CUDA library in-tree for sm_103a (nvcc, one object per file,
compiled in parallel, linked into ``_build/libdartree.so``)."""
from __future__ import annotations

import os
import platform
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build", platform.machine())
LIB = os.path.join(OUT_DIR, "libdartree.so")
# (source, extra flags, object name): the head kernels are built once per MMA N
_NS = (16, 32, 64, 128, 256)
SOURCES = ([("api.cu", [], "api.o"), ("select.cu", [], "select.o"),
            ("noalloc.cu", [], "noalloc.o"), ("variants.cu", [], "variants.o"), ("verify.cu", [], "verify.o"),
            ("head_rows.cu", [], "head_rows.o"), ("head_f32.cu", [], "head_f32.o")]
           + [("head_tc.cu", [f"-DDT_N={n}"], f"head_tc_{n}.o") for n in _NS]
           + [("head_simt.cu", [f"-DDT_N={n}"], f"head_simt_{n}.o") for n in _NS])
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-v", "-Wno-deprecated-gpu-targets"]


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(HERE, "..", "include", "dartree.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files if os.path.exists(f))


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB

    def compile_one(job) -> tuple[str, str]:
        src, extra, name = job
        obj = os.path.join(OUT_DIR, name)
        cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(min(len(SOURCES), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
