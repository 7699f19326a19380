"""Build libsplitkv.so in-tree with nvcc for sm_103a (GB300).

Each .cu translation unit compiles in parallel to an object under
``split_kv_flash_attn_gb300/_build/``; the objects link into
``split_kv_flash_attn_gb300/libsplitkv.so``.  The CUDA runtime is linked
statically, so the library needs no CUDA library path at load time.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libsplitkv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
         "-Xcudafe", "--diag_suppress=177"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (CUDA toolkit required to build libsplitkv.so)")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu*")) + glob.glob(os.path.join(CSRC, "*.h")) +
                  glob.glob(os.path.join(PKG, "..", "include", "*.h")) + [os.path.join(PKG, "exports.map")])


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    headers = [d for d in _deps() if not d.endswith(".cu")]
    jobs = []
    for src in _sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        if force or _stale(obj, [src] + headers):
            cmd = [cc, *ARCH, *FLAGS, "-c", src, "-o", obj]
            if ptxas_v:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append((src, cmd))
    if jobs:
        workers = max(1, min(len(jobs), os.cpu_count() or 4))
        with cf.ThreadPoolExecutor(workers) as ex:
            futs = {ex.submit(subprocess.run, cmd, capture_output=True, text=True): src for src, cmd in jobs}
            errors = []
            for fut in cf.as_completed(futs):
                res = fut.result()
                if verbose or ptxas_v:
                    sys.stderr.write(res.stderr)
                if res.returncode != 0:
                    errors.append(f"{futs[fut]}:\n{res.stderr}")
            if errors:
                raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in _sources()]
    if force or jobs or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        # export the C ABI only (skv_*): internal symbols stay local, so two
        # copies of the library in one process never share internal state
        exports = os.path.join(PKG, "exports.map")
        res = subprocess.run([cc, *ARCH, "-shared", "-Xlinker", f"--version-script={exports}", "-o", tmp, *objs],
                             capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("link failed:\n" + res.stderr)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_v="--ptxas-v" in sys.argv)
    print(LIB)
