"""Build the C-ABI library libdflash.so in-tree with nvcc (sm_103a only).

Each .cu file is compiled to an object in parallel, then linked into one
shared library under block_diffusion_drafter_inject_gb300/lib/.  The library
links the CUDA runtime statically and reaches the driver's tensor-map encoder
through the runtime's entry-point query, so it needs no libcuda at link time.
"""

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libdflash.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc():
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdflash.so")
    return p


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def portable_flags(flags, root=ROOT):
    """The compile flags with paths inside the checkout written relative to its
    root, so that they do not depend on where the repository sits."""
    out = []
    for f in flags:
        if os.path.isabs(f) and (f == root or f.startswith(root.rstrip(os.sep) + os.sep)):
            f = os.path.relpath(f, root)
        out.append(f)
    return out


def source_fingerprint(root=None):
    """Hash of the kernel sources, headers and compile flags (independent of the
    machine and of the checkout path): identifies the build a stored profile
    measurement belongs to.  `root` reads the sources of another checkout."""
    root = ROOT if root is None else root
    csrc = os.path.join(root, os.path.relpath(CSRC, ROOT))
    include = os.path.join(root, os.path.relpath(INCLUDE, ROOT))
    flags = [os.path.join(root, os.path.relpath(f, ROOT)) if f in (CSRC, INCLUDE) else f
             for f in FLAGS]
    h = hashlib.sha256()
    for d in (csrc, include):
        for f in sorted(os.listdir(d)):
            if f.endswith((".cu", ".cuh", ".h")):
                h.update(f.encode())
                h.update(open(os.path.join(d, f), "rb").read())
    h.update(" ".join(ARCH + portable_flags(flags, root)).encode())
    return h.hexdigest()


def _fingerprint():
    return source_fingerprint() + "|" + os.uname().machine


def build(force=False, verbose=False, extra_flags=()):
    """Compile libdflash.so if sources changed; returns its path."""
    os.makedirs(LIBDIR, exist_ok=True)
    stamp = os.path.join(LIBDIR, "libdflash.stamp")
    fp = _fingerprint() + "|" + " ".join(extra_flags)
    if not force and os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == fp:
        return LIB
    cc = nvcc()
    objdir = os.path.join(LIBDIR, "obj")
    os.makedirs(objdir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc] + ARCH + FLAGS + list(extra_flags) + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    srcs = sources()
    with ThreadPoolExecutor(len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = LIB + ".tmp"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(fp)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
