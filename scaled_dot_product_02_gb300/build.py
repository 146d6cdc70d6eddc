"""Build libsdpa.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit under csrc/ compiles in parallel; the objects link into
scaled_dot_product_02_gb300/libsdpa.so with the CUDA runtime linked statically
(the library only needs the NVIDIA driver at run time). The same sources
compiled with SDPA_ADDR_CHECK link into libsdpa_checked.so, the testing build
whose kernels test every computed global access against the call's buffers
(see sdpa_debug_address_report in include/sdpa.h).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libsdpa.so")
VARIANTS = {  # name: (object folder, library, extra nvcc flags)
    "normal": (BUILD, LIB, []),
    "checked": (os.path.join(PKG, "_build_checked"), os.path.join(PKG, "libsdpa_checked.so"), ["-DSDPA_ADDR_CHECK"]),
}
INCLUDE = os.path.join(os.path.dirname(PKG), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", f"-I{INCLUDE}"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers_mtime():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs.append(os.path.join(INCLUDE, "sdpa.h"))
    return max(os.path.getmtime(h) for h in hs)


def _compile(src: str, variant: str, verbose: bool) -> str:
    objdir, _, extra = VARIANTS[variant]
    obj = os.path.join(objdir, os.path.basename(src) + ".o")
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), _headers_mtime()):
        return obj
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj + ".tmp"]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def _link(variant: str, objs) -> str:
    _, lib, _ = VARIANTS[variant]
    if not os.path.exists(lib) or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


def build(verbose: bool = False, variants=("normal", "checked")) -> str:
    """Compile every translation unit of each variant in parallel and link the
    libraries; returns the path of libsdpa.so."""
    for v in variants:
        os.makedirs(VARIANTS[v][0], exist_ok=True)
    srcs = sources()
    jobs = [(s, v) for v in variants for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=min(os.cpu_count() or 8, len(jobs), 16)) as ex:
        objs = list(ex.map(lambda j: _compile(j[0], j[1], verbose), jobs))
    for v in variants:
        _link(v, [o for (s, vv), o in zip(jobs, objs) if vv == v])
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
