"""Build the in-tree CUDA library ``_lib/libsparse_engine.so`` for sm_103a.

Each translation unit under ``csrc/`` is compiled by nvcc in parallel, then
linked into one shared library against the shared CUDA runtime (the same
``libcudart.so.13`` PyTorch loads, found by soname, with the toolkit's lib64 as
the fallback run path).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB_NAME = "libsparse_engine.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cu", "quest_summary.cu", "quest_score.cu", "quest_topk.cu", "sparse_decode.cu", "mla_decode.cu", "quest_fused.cu",
           "decode_noalloc.cu", "snapkv.cu", "graph.cu"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _cuda_home(nvcc):
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def lib_path() -> str:
    return os.path.join(OUT_DIR, LIB_NAME)


def build(verbose: bool = False, ptxas_verbose: bool = False) -> str:
    nvcc = _nvcc()
    home = _cuda_home(nvcc)
    obj_dir = os.path.join(OUT_DIR, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    flags = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
             "-DNDEBUG"] + ARCH
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj] + flags
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_verbose:
        for _, err in results:
            if err:
                sys.stderr.write(err)
    out = lib_path()
    tmp = out + ".tmp"
    cmd = [nvcc, "-shared", "-o", tmp] + [o for o, _ in results] + ARCH + [
        "-cudart", "shared", "-Xlinker", f"-rpath,{os.path.join(home, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose=True, ptxas_verbose="-v" in sys.argv))
