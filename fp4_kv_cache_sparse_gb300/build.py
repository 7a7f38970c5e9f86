"""Build of the sm_103a library libmla.so (nvcc, in-tree, no cmake).

Each CUDA translation unit is compiled in parallel with
``-gencode arch=compute_103a,code=sm_103a -lineinfo -Xptxas -v``; the
ptxas report is parsed and the build FAILS if any kernel spills registers
(no switch turns this off).  The objects are linked into
``_build/libmla.so`` against the shared CUDA runtime.
"""
from __future__ import annotations

import concurrent.futures
import os
import re
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libmla.so")
SOURCES = ["api.cu", "metadata.cu", "decode.cu", "decode_pair.cu", "combine.cu", "dequant.cu", "noalloc.cu", "kv_write.cu"]
HEADERS = ["mla_device.cuh", "mla_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "--expt-relaxed-constexpr"]

_SPILL = re.compile(r"(\d+) bytes spill stores, (\d+) bytes spill loads")
_FUNC = re.compile(r"Compiling entry function '([^']+)'|Function properties for (\S+)")


class SpillError(RuntimeError):
    pass


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _inputs_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(HERE, "..", "include", "mla.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def _check_spills(src: str, log: str) -> list[str]:
    bad, current = [], None
    for line in log.splitlines():
        m = _FUNC.search(line)
        if m:
            current = m.group(1) or m.group(2)
        s = _SPILL.search(line)
        if s and (int(s.group(1)) or int(s.group(2))):
            bad.append(f"{src}: {current}: {line.strip()}")
    return bad


def refuse_spills(sources: list[str], logs: list[str]) -> None:
    """Raise SpillError naming every kernel whose ptxas report shows spill
    stores or loads (the library is then not linked)."""
    spills = []
    for src, log in zip(sources, logs):
        spills += _check_spills(src, log)
    if spills:
        raise SpillError("register spills (the build refuses them):\n" + "\n".join(spills))


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD, src.replace(".cu", ".o"))
    cmd = [nvcc(), *ARCH, *FLAGS, "-I", os.path.join(HERE, "..", "include"), "-c",
           os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _inputs_mtime():
        return LIB
    with concurrent.futures.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    report = [log for _, log in results]
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        f.write("\n".join(report))
    if verbose:
        print("\n".join(report))
    refuse_spills(SOURCES, report)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
