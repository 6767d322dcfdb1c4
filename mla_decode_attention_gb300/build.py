"""Builds the in-tree C-ABI library ``libmla_decode.so`` for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled in parallel with nvcc, then
linked into one shared library next to this file.  The build fails when any
kernel spills registers (the ptxas report of every kernel is checked, as the
FlashMLA build does after compiling; ``MLA_SKIP_REG_SPILL_CHECK=1`` skips
the check).  ``python -m
mla_decode_attention_gb300.build`` runs it.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import re
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libmla_decode.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-Xptxas", "-v", "-diag-suppress", "177"]


def _nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found")
    return path


def _sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(BUILD_DIR, src[:-3] + ".o")
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-c",
           os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


_ENTRY = re.compile(r"Compiling entry function '([^']+)'")
_SPILL = re.compile(r"(\d+) bytes spill stores, (\d+) bytes spill loads")


def spill_report(ptxas_log: str) -> list[str]:
    """Kernels that spill registers, one line each, from a ``-Xptxas -v`` log.

    Each ``Compiling entry function`` line names a kernel; the next
    ``bytes spill stores, ... bytes spill loads`` line gives its spills.
    """
    out = []
    entry = None
    for line in ptxas_log.splitlines():
        m = _ENTRY.search(line)
        if m:
            entry = m.group(1)
            continue
        m = _SPILL.search(line)
        if m and (int(m.group(1)) or int(m.group(2))):
            out.append(f"{entry}: {line.strip()}")
    return out


def build(verbose: bool = False) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = list(ex.map(_compile, _sources()))
    objs = [o for o, _ in results]
    log = "\n".join(l for _, l in results)
    with open(os.path.join(BUILD_DIR, "ptxas.log"), "w") as f:
        f.write(log)
    if verbose:
        print(log)
    spills = spill_report(log)
    if spills and os.environ.get("MLA_SKIP_REG_SPILL_CHECK") != "1":
        raise RuntimeError("register spilling detected, build failed (set "
                           "MLA_SKIP_REG_SPILL_CHECK=1 to skip this check):\n" + "\n".join(spills))
    lib = os.path.join(HERE, LIB_NAME)
    tmp = lib + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
