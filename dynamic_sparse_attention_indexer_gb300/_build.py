"""In-tree build of the C-ABI library ``libdsa_gb300.so`` for sm_103a, and of
``libdsa_probe.so`` (the peak-rate microbenchmarks the measurement reports its
roofline fractions against; not part of the dsa_* interface).

Each source is compiled by nvcc in parallel into ``_build/``, then linked
into the shared libraries beside this file.  A stamp of the sources, flags and
machine skips the build when nothing changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import platform
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdsa_gb300.so")
PROBE_LIB = os.path.join(PKG, "libdsa_probe.so")
PROBE_SOURCES = ["probe_peaks.cu"]
SOURCES = ["api.cpp", "kv_alloc.cpp", "k_index.cu", "k_topk.cu", "k_attn.cu", "k_misc.cu",
           "k_topk_static.cu", "k_prefix.cu", "k_dense.cu",
           "k_pselect.cu"]
HEADERS = ["common.cuh", "select.cuh", "internal.h", "attn_tile.cuh", "score_walk.cuh", "tc.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the DSA library needs the CUDA toolkit to build")


def _stamp() -> str:
    h = hashlib.sha256()
    for name in SOURCES + PROBE_SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    with open(os.path.join(ROOT, "include", "dsa.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(ARCH + FLAGS).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def _lib_matches_machine(path: str = LIB) -> bool:
    """The library exists and was linked for this machine (the tree may have
    been copied from a host of another architecture)."""
    if not os.path.exists(path):
        return False
    with open(path, "rb") as f:
        head = f.read(20)
    if head[:4] != b"\x7fELF":
        return False
    machine = int.from_bytes(head[18:20], "little")
    want = {"x86_64": 62, "aarch64": 183, "arm64": 183}.get(platform.machine())
    return want is None or machine == want


def is_current() -> bool:
    stamp_file = os.path.join(OUT_DIR, "stamp")
    if not _lib_matches_machine() or not _lib_matches_machine(PROBE_LIB) or not os.path.exists(stamp_file):
        return False
    with open(stamp_file) as f:
        return f.read().strip() == _stamp()


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and is_current():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(name):
        obj = os.path.join(OUT_DIR, name + ".o")
        cmd = [nvcc] + ARCH + FLAGS + ["-c", os.path.join(CSRC, name), "-o", obj]
        if name.endswith(".cu"):
            cmd += ["-Xptxas", "-v"] if verbose else []
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {name}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES) + len(PROBE_SOURCES)) as ex:
        results = dict(zip(SOURCES + PROBE_SOURCES, ex.map(compile_one, SOURCES + PROBE_SOURCES)))
    if verbose:
        for _, log in results.values():
            if log.strip():
                print(log)
    for lib, names in ((LIB, SOURCES), (PROBE_LIB, PROBE_SOURCES)):
        tmp = lib + ".tmp"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [results[n][0] for n in names]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    with open(os.path.join(OUT_DIR, "stamp"), "w") as f:
        f.write(_stamp())
    return LIB


def ensure_built() -> str:
    return build(force=False)


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
