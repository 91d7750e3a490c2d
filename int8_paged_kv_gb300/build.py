"""Build libpa_q8.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit under csrc/ compiles to an object in parallel, then
one link makes ``int8_paged_kv_gb300/libpa_q8.so``.  No torch, no cmake.
``python -m int8_paged_kv_gb300.build [-v]`` runs it (-v adds ptxas
register / spill reports).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpa_q8.so")
SOURCES = ["abi.cu", "writer.cu", "decode.cu", "decode_umma.cu", "decode_f32.cu", "decode_cq.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (looked at $NVCC, /usr/local/cuda/bin/nvcc, PATH)")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _flags_changed(stamp: str, key: str) -> bool:
    """True unless `stamp` records exactly this compiler command (`key`):
    objects built with other flags are stale whatever their times."""
    try:
        with open(stamp) as f:
            return f.read() != key
    except OSError:
        return True


def _record_flags(stamp: str, key: str) -> None:
    with open(stamp, "w") as f:
        f.write(key)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    headers.append(os.path.join(os.path.dirname(HERE), "include", "pa_q8.h"))
    cc = nvcc()
    include = os.path.join(os.path.dirname(HERE), "include")
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-I", include, "-Xcompiler", "-fPIC",
                    "-Xcompiler", "-O2"]
    flags += os.environ.get("PA_Q8_NVCC_FLAGS", "").split()
    # objects built with other flags (PA_Q8_NVCC_FLAGS) are stale whatever their times
    stamp = os.path.join(BUILD, "flags.txt")
    key = " ".join([cc] + flags)
    force = force or _flags_changed(stamp, key)
    if verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src: str) -> tuple[str, str]:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        if force or verbose or _stale(o, [s] + headers):
            r = subprocess.run([cc] + flags + ["-c", s, "-o", o], capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
            return o, r.stderr
        return o, ""

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    objs = [o for o, _ in results]
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    if force or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        r = subprocess.run([cc] + ARCH + ["-shared", "-o", tmp] + objs, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
        _record_flags(stamp, key)
    return LIB


if __name__ == "__main__":
    print(build(force="-f" in sys.argv, verbose="-v" in sys.argv))
