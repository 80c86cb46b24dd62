"""In-tree build of the CUDA library (libattn) for sm_103a with nvcc.

Each translation unit compiles in parallel to an object file; the objects are
linked into one shared library under ``_build/``, named by a hash of the sources
and flags, so a stale library is never loaded.
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")

SOURCES = [
    "attn_api.cu",
    "attn_inst_d64_dv64.cu",
    "attn_inst_d64_dv128.cu",
    "attn_inst_d128_dv64.cu",
    "attn_inst_d128_dv128.cu",
    "attn_pair_inst.cu",
    "attn_pair_dense_inst.cu",
    "attn_pair_key_inst.cu",
    "attn_static_scratch.cu",
    "attn_host_stream.cu",
    "attn_bwd_inst_d64_dv64.cu",
    "attn_bwd_inst_d64_dv128.cu",
    "attn_bwd_inst_d128_dv64.cu",
    "attn_bwd_inst_d128_dv128.cu",
]
HEADERS = ["attn_fwd_kernel.cuh", "attn_fwd_pair_kernel.cuh", "attn_merge_kernel.cuh", "attn_bwd_kernel.cuh", "ptx.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden"]


def nvcc() -> str:
    cand = shutil.which("nvcc")
    if cand:
        return cand
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    if os.path.exists(path):
        return path
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn")


def source_hash(extra_flags=()) -> str:
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    with open(os.path.join(INCLUDE, "attn.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(ARCH + NVCC_FLAGS + list(extra_flags)).encode())
    return h.hexdigest()[:16]


def library_path(extra_flags=()) -> str:
    return os.path.join(BUILD_DIR, f"libattn_{source_hash(extra_flags)}.so")


def build(verbose: bool = False, extra_flags=(), jobs: int | None = None) -> str:
    """Compile and link libattn if the current sources have no library yet; return its path."""
    so = library_path(extra_flags)
    if os.path.exists(so):
        return so
    os.makedirs(BUILD_DIR, exist_ok=True)
    tag = os.path.basename(so)[len("libattn_"):-3]
    obj_dir = os.path.join(BUILD_DIR, f"obj_{tag}_{os.getpid()}")
    os.makedirs(obj_dir, exist_ok=True)
    exe = nvcc()

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
        cmd = [exe, *ARCH, *NVCC_FLAGS, *extra_flags, "-I", INCLUDE, "-I", CSRC, "-c",
               os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)
        return obj

    workers = jobs or min(len(SOURCES), os.cpu_count() or 1)
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = so + f".tmp{os.getpid()}"
    cmd = [exe, *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, so)
    shutil.rmtree(obj_dir, ignore_errors=True)
    return so
