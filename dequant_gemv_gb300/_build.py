"""In-tree build of libq4nx.so for sm_103a (nvcc, one -gencode, parallel TUs).

``python dequant_gemv_gb300/_build.py`` or ``build()`` compiles every
``csrc/*.cu`` into ``_objs/`` and links ``libq4nx.so`` next to this file.
Objects are rebuilt only when a source or header is newer.  No cmake.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJS = os.path.join(PKG, "_objs")
LIB = os.path.join(PKG, "libq4nx.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fno-strict-aliasing"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libq4nx.so")


def _headers() -> list[str]:
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(OBJS, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = _headers()
    jobs = []
    for src in sources:
        obj = os.path.join(OBJS, os.path.basename(src)[:-3] + ".o")
        if _stale(obj, [src] + headers) or ptxas_info:
            cmd = [nvcc, *ARCH, *FLAGS, "-c", src, "-o", obj]
            if ptxas_info:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append((src, cmd))

    def run(job):
        src, cmd = job
        p = subprocess.run(cmd, capture_output=True, text=True)
        return src, p.returncode, p.stdout + p.stderr

    if jobs:
        with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
            results = list(ex.map(run, jobs))
        failed = [(s, out) for s, rc, out in results if rc != 0]
        for s, rc, out in results:
            if verbose or ptxas_info or rc != 0:
                sys.stderr.write(f"== {os.path.basename(s)} (rc={rc})\n{out}")
        if failed:
            raise RuntimeError("nvcc failed on: " + ", ".join(os.path.basename(s) for s, _ in failed))
    objs = [os.path.join(OBJS, os.path.basename(s)[:-3] + ".o") for s in sources]
    if _stale(LIB, objs) or jobs:
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError("link of libq4nx.so failed:\n" + p.stdout + p.stderr)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv))
