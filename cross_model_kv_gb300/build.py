"""Build libkvb.so in-tree with nvcc for sm_103a (GB300).

Each translation unit under csrc/ is compiled in parallel, then linked with
the static CUDA runtime into cross_model_kv_gb300/_lib/libkvb.so.  Nothing is
installed outside the package directory.  build(checked=True) makes the
checked variant, libkvb_checked.so (-DKVB_CHECK_BOUNDS=1: index checks on the
hot kernels' CUDA-core global accesses, failures reported as KVB_ERR_CUDA),
which the binding loads instead when KVB_LIBRARY=checked.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
OBJ_DIR = os.path.join(OUT_DIR, "obj")
LIB_PATH = os.path.join(OUT_DIR, "libkvb.so")
CHECKED_OBJ_DIR = os.path.join(OUT_DIR, "obj_checked")
CHECKED_LIB_PATH = os.path.join(OUT_DIR, "libkvb_checked.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
              "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(src: str, verbose: bool, ptxas_v: bool, checked: bool = False) -> tuple[str, str]:
    obj = os.path.join(CHECKED_OBJ_DIR if checked else OBJ_DIR, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *(["-DKVB_CHECK_BOUNDS=1"] if checked else []), "-c", src, "-o", obj]
    if ptxas_v:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return obj, (r.stdout + r.stderr) if (verbose or ptxas_v) else ""


def _stale(srcs: list[str], lib: str = LIB_PATH) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "kvb.h"), __file__]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False, checked: bool = False) -> str:
    """Compile and link libkvb.so (or libkvb_checked.so) if any source changed; return its path."""
    srcs = sources()
    lib_path = CHECKED_LIB_PATH if checked else LIB_PATH
    if not force and not ptxas_v and not _stale(srcs, lib_path):
        return lib_path
    os.makedirs(CHECKED_OBJ_DIR if checked else OBJ_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose, ptxas_v, checked), srcs))
    for _, log in results:
        if log:
            sys.stderr.write(log)
    tmp = lib_path + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for o, _ in results], "-ldl", "-lpthread",
           "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_v="--ptxas-v" in sys.argv,
                checked="--checked" in sys.argv))
