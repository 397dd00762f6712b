"""Builds libdflash_gb300.so in-tree with nvcc for sm_103a (GB300) only.

Translation units are compiled in parallel, then linked with nvcc -shared. The output
lands in speculative_decoding_draft_rmsnorm_gb300/_lib/; objects go to _build/.

A second library, libdflash_gb300_waittest.so, is built from the same sources with
DFLASH_WAIT_TEST defined: device waits give up after 5 ms instead of 2 s, and a hook can
withhold one V tile's copy, so that a test can watch a bounded wait run out and the
kernel unwind. Only the tests load it; the package loads the product library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_NAME = "libdflash_gb300.so"
LIB_PATH = os.path.join(LIB_DIR, LIB_NAME)
SOURCES = ["api.cu", "attention.cu", "norm_rope.cu", "noalloc.cu", "draft_step.cu"]
HEADERS = ["ptx.cuh", "internal.h", "norm_rope.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "-DDFLASH_BUILD"]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build the library")
    return p


WAIT_TEST_LIB_PATH = os.path.join(LIB_DIR, "libdflash_gb300_waittest.so")
# (library, extra nvcc flags, object folder)
TARGETS = [(LIB_PATH, [], OBJ_DIR),
           (WAIT_TEST_LIB_PATH, ["-DDFLASH_WAIT_TEST"], os.path.join(OBJ_DIR, "waittest"))]


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "dflash.h"))
    return files


def up_to_date(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Builds both libraries (every translation unit of both in one parallel pass) and
    returns the product library's path."""
    todo = [t for t in TARGETS if force or not up_to_date(t[0])]
    if not todo:
        return LIB_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    cc = nvcc()

    def compile_one(job) -> str:
        src, extra, obj_dir = job
        obj = os.path.join(obj_dir, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} {' '.join(extra)}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    jobs = []
    for _, extra, obj_dir in todo:
        os.makedirs(obj_dir, exist_ok=True)
        jobs += [(src, extra, obj_dir) for src in SOURCES]
    workers = max(1, min(len(jobs), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        objs = list(ex.map(compile_one, jobs))
    for i, (path, _, _) in enumerate(todo):
        tmp = path + f".tmp{os.getpid()}"
        mine = objs[i * len(SOURCES):(i + 1) * len(SOURCES)]
        r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *mine, "-lcudart"], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, path)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
