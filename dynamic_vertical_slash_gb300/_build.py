"""Compiles the CUDA library (csrc/*.cu) for sm_103a into _lib/libvs.so.

One -gencode, translation units compiled in parallel, no CMake.  The result
stays in the source tree so that every process loads the same in-tree file.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INC = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libvs.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr", "-I", INC]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _digest() -> str:
    """Build stamp: the sources' digest plus the compiler flags (paths taken
    out, so that the stamp does not depend on where the tree lives)."""
    h = hashlib.sha256(source_digest().encode())
    h.update(" ".join(ARCH + [("<include>" if f == INC else f) for f in FLAGS]).encode())
    return h.hexdigest()


# The translation unit of each traced kernel name (all headers count for all).
KERNEL_SOURCES = {
    "fwd": "vs_attn_fwd.cu", "bwd_dq": "vs_attn_bwd.cu", "bwd_dkv_slash": "vs_attn_bwd.cu",
    "bwd_dkv_bar": "vs_attn_bwd.cu", "bwd_prep": "vs_attn_bwd.cu", "index": "vs_index.cu",
    "striped_permute": "vs_permute.cu", "ring_work": "vs_ringwork.cu",
}


def source_digest(kernel: str = None) -> str:
    """SHA-256 of source contents and file names only (no paths, no flags):
    every file under csrc/ and include/, or, for a traced kernel name, its
    translation unit plus every header.  A profile of a kernel records this
    digest; it stays valid while the digest is unchanged."""
    files = sorted(glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INC, "*.h")))
    if kernel is not None:
        tu = KERNEL_SOURCES.get(kernel, "vs_estimate.cu" if kernel.startswith("est_") else None)
        if tu is None:
            raise KeyError(kernel)
        files = [f for f in files if not f.endswith(".cu") or os.path.basename(f) == tu]
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False) -> str:
    stamp = os.path.join(OUT_DIR, "build.sha256")
    digest = _digest()
    if not force and os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == digest:
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(OUT_DIR, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc] + ARCH + FLAGS + ["-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        for obj, log in ex.map(compile_one, _sources()):
            objs.append(obj)
            if verbose and log:
                print(log)
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    with open(stamp, "w") as fh:
        fh.write(digest)
    return LIB


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
