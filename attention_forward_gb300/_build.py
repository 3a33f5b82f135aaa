"""Builds libfa_gb300.so in-tree from csrc/ with nvcc for sm_103a.

Each translation unit is compiled in its own nvcc process (in parallel), then
the objects are linked into one shared library against the shared CUDA
runtime, so the library and PyTorch use the same runtime instance when both
are loaded.  ``python -m attention_forward_gb300._build`` builds it.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_objs")
LIB = os.path.join(PKG, "libfa_gb300.so")
PTXAS_LOG = os.path.join(OBJ, "ptxas.log")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xptxas", "-v", "--expt-relaxed-constexpr",
                     f"-I{os.path.join(ROOT, 'include')}"]
SOURCES = ["fa_prefill_d128.cu", "fa_prefill_d64.cu", "fa_prefill_d64x3.cu", "fa_prefill_pair.cu",
           "fa_decode.cu", "fa_api.cu", "fa_noalloc.cu", "fa_diag.cu"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _cuda_lib_dir() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc()))),
                        "lib64")


def _fingerprint() -> str:
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)):
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    with open(os.path.join(ROOT, "include", "fa.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(NVCC_FLAGS).encode())
    return h.hexdigest()


def _compile(src: str, obj_dir: str = OBJ, defines=()) -> tuple[str, str]:
    obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *NVCC_FLAGS, *[f"-D{d}" for d in defines], "-c",
           os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, defines=(),
          variant: str | None = None) -> str:
    """Compile and link the library unless an up-to-date build exists.

    ``variant`` with ``defines`` (macro names, optionally NAME=VALUE) builds
    another copy of the same sources with those macros set, into
    ``_variants/libfa_gb300_<variant>.so``: the alternative arms of paired
    measurements (bench.py --paired).  The in-tree library is unaffected."""
    defines = tuple(defines)
    obj_dir, lib = OBJ, LIB
    if variant is not None:
        obj_dir = os.path.join(PKG, "_variants", f"objs_{variant}")
        lib = os.path.join(PKG, "_variants", f"libfa_gb300_{variant}.so")
    os.makedirs(obj_dir, exist_ok=True)
    stamp = os.path.join(obj_dir, "fingerprint")
    fp = _fingerprint() + " ".join(defines)
    if (not force and os.path.exists(lib) and os.path.exists(stamp)
            and open(stamp).read() == fp):
        return lib
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, obj_dir, defines), SOURCES))
    with open(os.path.join(obj_dir, "ptxas.log"), "w") as f:
        for (obj, log), src in zip(results, SOURCES):
            f.write(f"==== {src}\n{log}\n")
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "--cudart", "shared", "-o", tmp,
           *[o for o, _ in results], f"-L{_cuda_lib_dir()}",
           "-Xlinker", f"-rpath,{_cuda_lib_dir()}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(fp)
    if verbose:
        print(open(os.path.join(obj_dir, "ptxas.log")).read())
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
