"""Build ``libspark_attn.so`` in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled in parallel into
``_build/`` and linked into ``libspark_attn.so`` next to this file.  The
library is rebuilt when a source or header is newer than it (or ``force``).
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB_NAME = "libspark_attn.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)

SOURCES = ["api.cu", "proj.cu", "attn.cu", "stack.cu", "noalloc.cu", "mma.cu", "mlp.cu", "layer_api.cu", "attn_chunk.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                 "-Xcompiler", "-Wall", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libspark_attn.so")


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)
             if f.endswith((".cu", ".cuh", ".h"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return files


STAMP = os.path.join(BUILD, "flags.txt")


def _extra_flags() -> list[str]:
    """Extra nvcc flags from SPARK_NVCC_FLAGS (e.g. tuning -D overrides)."""
    return os.environ.get("SPARK_NVCC_FLAGS", "").split()


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    old = open(STAMP).read() if os.path.exists(STAMP) else ""
    if old != " ".join(_extra_flags()):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _run(cmd: list[str], verbose: bool) -> None:
    if verbose:
        print(" ".join(cmd), flush=True)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"command failed ({res.returncode}): {' '.join(cmd)}\n"
                           f"{res.stdout}\n{res.stderr}")
    if verbose and (res.stdout or res.stderr):
        print(res.stdout + res.stderr, flush=True)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link the library if needed; return its path."""
    if not force and not ptxas_info and not _stale():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + _extra_flags()
    objs = []
    cmds = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(obj)
        cmds.append([nvcc] + CFLAGS + extra + ["-c", os.path.join(CSRC, src), "-o", obj])
    with cf.ThreadPoolExecutor(max_workers=len(cmds)) as ex:
        list(ex.map(lambda c: _run(c, verbose or ptxas_info), cmds))
    tmp = LIB_PATH + ".tmp"
    _run([nvcc] + ARCH + ["-shared", "-o", tmp] + objs, verbose)
    os.replace(tmp, LIB_PATH)
    with open(STAMP, "w") as f:
        f.write(" ".join(_extra_flags()))
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
