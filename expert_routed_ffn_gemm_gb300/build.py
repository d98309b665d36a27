"""Build step of libmoe.so: every CUDA source under csrc/ compiled for sm_103a
with nvcc (in parallel), linked into one shared library with the CUDA runtime
linked statically (the library loads without a GPU driver; CUDA calls then fail
with a status code).  The same sources compiled with -DMOE_DEBUG make
libmoe_debug.so, whose kernels check the indices they take from the dispatch
(see kernels.cuh)."""
from __future__ import annotations

import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
LIB_DIR = os.path.join(PKG, "lib")
HEADER = os.path.join(ROOT, "include", "moe.h")
VARIANTS = {
    # name: (object directory, library, extra flags)
    "release": (os.path.join(ROOT, "_build", "obj"), os.path.join(LIB_DIR, "libmoe.so"), []),
    "debug": (os.path.join(ROOT, "_build", "obj_debug"), os.path.join(LIB_DIR, "libmoe_debug.so"), ["-DMOE_DEBUG"]),
}
LIB_PATH = VARIANTS["release"][1]
DEBUG_LIB_PATH = VARIANTS["debug"][1]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-Xptxas", "-warn-spills"] + ARCH


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hdrs + [HEADER, os.path.abspath(__file__)]


def _stale(target: str, inputs: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(p) > t for p in inputs)


def _run(cmd, verbose):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr)


def build(force: bool = False, verbose: bool = False, variants=("release", "debug")) -> str:
    """Compile and link the named library variants where any input is newer
    (every translation unit of every variant in one parallel pool); returns
    the release library's path."""
    os.makedirs(LIB_DIR, exist_ok=True)
    nvcc = _nvcc()
    deps = _deps()
    srcs = sources()
    jobs, links = [], []
    for v in variants:
        obj_dir, lib, extra = VARIANTS[v]
        os.makedirs(obj_dir, exist_ok=True)
        objs = []
        for s in srcs:
            o = os.path.join(obj_dir, os.path.basename(s)[:-3] + ".o")
            objs.append(o)
            if force or _stale(o, [s] + deps):
                jobs.append([nvcc] + NVCC_FLAGS + extra + ["-c", s, "-o", o])
        links.append((lib, objs))
    with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        list(ex.map(lambda c: _run(c, verbose), jobs))
    for lib, objs in links:
        if force or _stale(lib, objs):
            tmp = lib + f".{os.getpid()}.tmp"
            _run([nvcc, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"], verbose)
            os.replace(tmp, lib)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
