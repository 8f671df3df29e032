"""Builds libtreeverify.so in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` compiles to an object in ``_build/`` in
parallel; the objects link into ``libtreeverify.so`` next to this file.  The
CUDA runtime is linked statically and the driver API is reached through the
runtime's entry-point query, so the library loads on machines without a GPU
driver (symbol checks) and needs only the driver at run time.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libtreeverify.so")
# development build with test hooks (-DTV_TEST_HOOKS): a settable wait limit
# and a withheld TMA load in the tensor-core attention kernels, so a test can
# run their timeout exit; never loaded unless TREEVERIFY_LIB names it
DEV_BUILD = os.path.join(BUILD, "dev")
DEV_LIB = os.path.join(DEV_BUILD, "libtreeverify_dev.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
          "-I" + os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]


def nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found")
    return exe


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _compile(src, extra, outdir=BUILD):
    obj = os.path.join(outdir, os.path.basename(src) + ".o")
    cmd = [nvcc(), *ARCH, *COMMON, *extra, "-c", src, "-o", obj]
    if src.endswith(".cpp"):
        cmd[1:1] = ["-x", "cu"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose=False, extra=None, jobs=None, dev=False):
    """Compile every source and link libtreeverify.so (``dev``: the test-hook
    build, DEV_LIB); returns the library's path."""
    outdir, lib_path = (DEV_BUILD, DEV_LIB) if dev else (BUILD, LIB)
    os.makedirs(outdir, exist_ok=True)
    extra = list(extra or []) + (["-DTV_TEST_HOOKS"] if dev else [])
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=jobs or min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, extra, outdir), srcs))
    objs = [o for o, _ in results]
    if verbose:
        for (o, err) in results:
            if err.strip():
                print(err, file=sys.stderr)
    tmp = lib_path + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    args = sys.argv[1:]
    print(build(verbose=True, extra=args))
