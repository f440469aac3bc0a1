"""Build the CUDA library ``libxqa_gb300.so`` in-tree with nvcc (sm_103a).

Each translation unit compiles in parallel; the link is plain ``nvcc
-shared``.  No torch headers are involved: the library's interface is the C
ABI of include/xqa.h.
"""

from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import platform
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libxqa_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "--cudart", "shared", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC,
         "--expt-relaxed-constexpr"]


def nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return exe


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


STAMP = LIB + ".sha256"


def source_files():
    """Every file the library is built from: csrc/ and the public header."""
    files = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h")))
    files.append(os.path.join(INCLUDE, "xqa.h"))
    return files


def source_digest(files=None):
    """SHA-256 over the sources' names and contents, the compiler flags and the
    host machine: the library is rebuilt whenever any of them changes, whatever
    the files' modification times say."""
    h = hashlib.sha256()
    for f in files if files is not None else source_files():
        h.update(os.path.basename(f).encode() + b"\0")
        with open(f, "rb") as fh:
            h.update(fh.read())
        h.update(b"\0")
    h.update(" ".join(ARCH + FLAGS).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def is_current(lib, stamp, digest):
    """True when `lib` exists and `stamp` records that it was built from `digest`."""
    if not (os.path.exists(lib) and os.path.exists(stamp)):
        return False
    with open(stamp) as fh:
        return fh.read().strip() == digest


def _compile(src, verbose):
    obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force=False, verbose=False):
    """Compile every .cu under csrc/ and link libxqa_gb300.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    digest = source_digest()
    if not force and is_current(LIB, STAMP, digest):
        return LIB
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose), srcs))
    if verbose:
        for obj, log in results:
            print(log)
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = [nvcc(), *ARCH, "-shared", "--cudart", "shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP + f".{os.getpid()}.tmp", "w") as fh:
        fh.write(digest + "\n")
    os.replace(STAMP + f".{os.getpid()}.tmp", STAMP)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
