"""Compile librot.so (the C-ABI library) in-tree for sm_103a with nvcc.

Each translation unit compiles in parallel into _build/, then one link step
writes matrix_optimizer_step_rot_gb300/librot.so.  Rebuilds only what changed
(by modification time against the object file and the shared headers).
"""

from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "librot.so")
# the bounds-checked variant (ROT_CHECK: guard regions around every workspace
# slice, checked after each micro-group; include/rot_testing.h)
BUILD_CHECK = os.path.join(PKG, "_build_check")
LIB_CHECK = os.path.join(PKG, "librot_check.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off",
              "-I", INCLUDE,
              "-I", CSRC, "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cu", ".cpp")))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return hs + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]


def build(verbose: bool = False, extra_flags=None, check: bool = False) -> str:
    """Build librot.so (check: the bounds-checked librot_check.so) if needed;
    returns its path.  Raises on compiler errors."""
    build_dir, lib = (BUILD_CHECK, LIB_CHECK) if check else (BUILD, LIB)
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = NVCC_FLAGS + (["-DROT_CHECK"] if check else []) + list(extra_flags or [])
    newest_header = max(os.path.getmtime(h) for h in _headers())
    jobs = []
    for src in _sources():
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        stale = (not os.path.exists(obj) or os.path.getmtime(obj) < os.path.getmtime(src)
                 or os.path.getmtime(obj) < newest_header)
        cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
        if src.endswith(".cu"):
            cmd += ["-Xptxas", "-v"] if verbose else []
        jobs.append((stale, cmd, obj))

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    stale_cmds = [c for s, c, _ in jobs if s]
    if stale_cmds:
        with ThreadPoolExecutor(max_workers=min(8, len(stale_cmds))) as ex:
            for cmd, r in ex.map(run, stale_cmds):
                if verbose and r.stderr:
                    sys.stderr.write(r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    objs = [o for _, _, o in jobs]
    if stale_cmds or not os.path.exists(lib):
        cmd = [nvcc, *ARCH, "-shared", "-o", lib + ".tmp", *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
