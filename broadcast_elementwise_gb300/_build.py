"""Build libebin.so (the C-ABI engine) in-tree for sm_103a.

Every kernel translation unit is compiled once per element class
(-DEBIN_DT=0..12) so the objects build in parallel; only objects older
than their sources are rebuilt.  No cmake, one -gencode.
"""
from __future__ import annotations

import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(PKG, "_build", platform.machine())
LIB = os.path.join(PKG, "libebin.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
GROUPS = ["arith", "mod", "pow", "cmp", "logic", "chan", "ext", "tern", "powmix"]
N_DT = 13
# -fmad=false: no multiply-add contraction anywhere; the kernels also use the
# _rn intrinsics explicitly.  No fast-math.
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-Xcompiler", "-fPIC",
              "-I" + INCLUDE, "-I" + CSRC]


def _elf_matches_host(path: str) -> bool:
    """True if the shared object at `path` was built for this machine's CPU."""
    import platform
    import struct
    want = {"x86_64": 62, "aarch64": 183, "arm64": 183}.get(platform.machine())
    try:
        with open(path, "rb") as f:
            head = f.read(20)
        return want is None or struct.unpack("<H", head[18:20])[0] == want
    except (OSError, struct.error):
        return False


def nvcc_path() -> str:
    cand = [os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"]
    for c in cand:
        p = os.path.join(c, "bin", "nvcc") if c else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found: the engine needs the CUDA 13 toolkit to build")
    return p


def _headers():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))] + \
        [os.path.join(INCLUDE, "ebin.h")]


def _stale(obj: str, deps) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def _jobs():
    nvcc = nvcc_path()
    heads = _headers()
    jobs = []
    host_src = os.path.join(CSRC, "ebin_host.cpp")
    host_obj = os.path.join(OBJDIR, "ebin_host.o")
    jobs.append((host_obj, [host_src] + heads,
                 [nvcc, *ARCH, *NVCC_FLAGS, "-c", host_src, "-o", host_obj]))
    noalloc_src = os.path.join(CSRC, "ebin_noalloc.cu")
    noalloc_obj = os.path.join(OBJDIR, "ebin_noalloc.o")
    jobs.append((noalloc_obj, [noalloc_src] + heads,
                 [nvcc, *ARCH, *NVCC_FLAGS, "-c", noalloc_src, "-o", noalloc_obj]))
    for g in GROUPS:
        src = os.path.join(CSRC, "k_%s.cu" % g)
        for dt in range(N_DT):
            obj = os.path.join(OBJDIR, "k_%s_%d.o" % (g, dt))
            jobs.append((obj, [src] + heads,
                         [nvcc, *ARCH, *NVCC_FLAGS, "-DEBIN_DT=%d" % dt, "-c", src, "-o", obj]))
    return nvcc, jobs


def build(force: bool = False, jobs: int | None = None, verbose: bool = False) -> str:
    """Compile and link libebin.so next to this file; returns its path."""
    os.makedirs(OBJDIR, exist_ok=True)
    nvcc, work = _jobs()
    todo = [(o, cmd) for o, deps, cmd in work if force or _stale(o, deps)]

    def run(item):
        obj, cmd = item
        tmp = obj + ".tmp%d.o" % os.getpid()
        cmd = cmd[:-1] + [tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (obj, " ".join(cmd), r.stderr))
        os.replace(tmp, obj)
        if verbose:
            sys.stderr.write("built %s\n" % os.path.basename(obj))

    if todo:
        n = jobs or max(1, min(len(todo), os.cpu_count() or 1))
        with ThreadPoolExecutor(n) as ex:
            list(ex.map(run, todo))
    objs = [o for o, _, _ in work]
    if force or todo or _stale(LIB, objs) or not _elf_matches_host(LIB):
        cuda_lib = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "lib64")
        tmp = LIB + ".tmp%d" % os.getpid()
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", "-rpath," + cuda_lib]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
