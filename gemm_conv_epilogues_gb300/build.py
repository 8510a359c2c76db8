"""Builds libtf_epilogue.so in-tree with nvcc for sm_103a (GB300).

Each translation unit under csrc/ is compiled in parallel, then linked into
one shared library next to this file.  No CMake, no torch extension
machinery: the library is plain C ABI (include/tf_epilogue.h).
"""
from __future__ import annotations

import concurrent.futures
import glob
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libtf_epilogue.so")
BUILD_DIR = os.path.join(PKG, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC] + ARCH


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtf_epilogue.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def _fingerprint() -> str:
    h = hashlib.sha256()
    for f in _sources() + _headers():
        h.update(f.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(NVCC_FLAGS).encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def build_library(force: bool = False, verbose: bool = False) -> str:
    """Compile and link if the sources changed since the last build; return the .so path.
    Concurrent callers (parallel test workers) serialise on a lock file."""
    import fcntl
    os.makedirs(BUILD_DIR, exist_ok=True)
    with open(os.path.join(BUILD_DIR, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        return _build_locked(force, verbose)


def _build_locked(force: bool, verbose: bool) -> str:
    stamp = LIB + ".stamp"
    fp = _fingerprint()
    if not force and os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == fp:
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
        cmd = [cc] + NVCC_FLAGS + ["-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
        return obj, r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, _sources()))
    if verbose:
        for _, err in results:
            if err.strip():
                print(err)
    tmp = LIB + f".tmp{os.getpid()}"
    r = subprocess.run([cc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as fh:
        fh.write(fp)
    return LIB


def resource_report() -> str:
    """Registers, spills and static shared memory of every kernel, from
    ptxas -v of a fresh compile (nothing is linked or installed), as a
    markdown table; kernels named by their source-level template."""
    import re
    import subprocess as sp
    import tempfile
    cc = nvcc()
    rows = []
    with tempfile.TemporaryDirectory() as tmp:
        for src in _sources():
            r = sp.run([cc] + NVCC_FLAGS + ["-Xptxas=-v", "-c", src, "-o", os.path.join(tmp, "x.o")],
                       capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(r.stderr)
            fn = None
            for line in r.stderr.splitlines():
                m = re.search(r"Compiling entry function '([^']+)'", line)
                if m:
                    fn = m.group(1)
                    spill = regs = smem = None
                    continue
                m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
                if m and fn:
                    spill = f"{m.group(1)}/{m.group(2)}"
                m = re.search(r"Used (\d+) registers(?:.*?(\d+) bytes smem)?", line)
                if m and fn:
                    regs, smem = m.group(1), m.group(2) or "0"
                    dm = sp.run(["c++filt", fn], capture_output=True, text=True).stdout.strip()
                    dm = dm.replace("tf::(anonymous namespace)::", "").replace("void ", "")
                    dm = dm[:dm.rindex(">(") + 1] if ">(" in dm else dm.split("(")[0]   # drop the parameter list
                    rows.append((os.path.basename(src), dm, regs, spill or "0/0", smem))
                    fn = None
    out = ["| file | kernel | registers | spill stores/loads (bytes) | static smem (bytes) |",
           "|---|---|---:|---:|---:|"]
    out += [f"| {f} | `{k}` | {r} | {sp_} | {sm} |" for f, k, r, sp_, sm in rows]
    return "\n".join(out)


if __name__ == "__main__":
    import sys
    if "--resources" in sys.argv:
        print(resource_report())
    else:
        print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))
