"""Builds librs.so (the CUDA library) in-tree with nvcc for sm_103a.

The translation units compile in parallel, then link into one shared library
against the shared CUDA runtime (the same one PyTorch loads).
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "librs.so")
SOURCES = ["rs_api.cu", "rs_replay.cu", "rs_replay_m2.cu", "rs_replay_gdn.cu", "rs_replay_kda.cu", "rs_replay_direct.cu", "rs_eager.cu",
           "rs_small.cu", "rs_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build librs")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _stale(out: str) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "rs.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(out: str = LIB, defines: list[str] | None = None, force: bool = False, verbose: bool = False) -> str:
    """Compile and link librs.so; returns its path.  ``defines`` adds -D flags."""
    if not force and not defines and not _stale(out):
        return out
    nvcc = _nvcc()
    objdir = os.path.join(os.path.dirname(out), "_build")
    os.makedirs(objdir, exist_ok=True)
    flags = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    flags += [f"-D{d}" for d in (defines or [])]
    tag = "_".join(d.replace("=", "") for d in (defines or [])) or "default"

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, f"{os.path.splitext(src)[0]}.{tag}.o")
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "--cudart=shared", "-o", tmp, *objs,
           "-Xlinker", f"-rpath={_cuda_lib_dir(nvcc)}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
