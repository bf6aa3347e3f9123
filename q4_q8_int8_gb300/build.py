"""Build libmmq.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit under csrc/ is compiled in parallel, then linked into
q4_q8_int8_gb300/lib/libmmq.so with the static CUDA runtime (no libcuda link:
the driver entry points are fetched at run time, so the library also loads
on a machine without a GPU).
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "libmmq.so")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")

NVCC = os.environ.get("NVCC", shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# No fast-math anywhere: the quantize prepass must match IEEE division and
# roundf bit for bit, and denormals are kept (-ftz=false).
CUFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-ftz=false",
           "-prec-div=true", "-prec-sqrt=true", "-fmad=true", "-I", INCLUDE]
CXXFLAGS = ["-O2", "-std=c++17", "-fPIC", "-I", INCLUDE]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cu", ".cpp")))


def _digest():
    h = hashlib.sha256()
    headers = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith((".h", ".cuh"))]
    for p in sources() + headers:
        h.update(p.encode())
        with open(p, "rb") as f:
            h.update(f.read())
    with open(os.path.join(INCLUDE, "mmq.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(ARCH + CUFLAGS + CXXFLAGS).encode())
    return h.hexdigest()


def _compile(src, obj, verbose):
    if src.endswith(".cu"):
        cmd = [NVCC, *ARCH, *CUFLAGS, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
    else:
        cmd = ["g++", *CXXFLAGS, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(LIBDIR, exist_ok=True)
    stamp = os.path.join(LIBDIR, "libmmq.stamp")
    dig = _digest()
    import platform
    dig += platform.machine()
    if not force and os.path.exists(LIB) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read() == dig:
                return LIB
    objdir = os.path.join(LIBDIR, "obj")
    os.makedirs(objdir, exist_ok=True)
    srcs = sources()
    objs = [os.path.join(objdir, os.path.basename(s) + ".o") for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        logs = list(ex.map(lambda so: _compile(so[0], so[1], verbose), zip(srcs, objs)))
    if verbose:
        for s, l in zip(srcs, logs):
            if l.strip():
                print(f"== {os.path.basename(s)}\n{l}", file=sys.stderr)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp, "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(dig)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
