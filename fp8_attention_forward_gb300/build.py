"""Builds libfa8.so (the C-ABI library) in-tree for sm_103a with nvcc.

Each translation unit under csrc/ is compiled in parallel; the objects are linked into
``_build/libfa8.so``.  ``python -m fp8_attention_forward_gb300.build`` runs it.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libfa8.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(ptxas_verbose: bool):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]
    if ptxas_verbose:
        f += ["-Xptxas", "-v"]
    return f


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
                  [os.path.join(ROOT, "include", "fa8.h")])


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _sources() + _headers() + [__file__])


def build(force: bool = False, ptxas_verbose: bool = False, jobs: int | None = None,
          out_dir: str | None = None, defines=(), src_dir: str | None = None) -> str:
    """Compiles csrc/*.cu and links libfa8.so into ``out_dir`` (default: the in-tree
    _build/); ``defines`` are extra -D macros (e.g. FA8_TRACE for the pipeline trace);
    ``src_dir`` compiles another copy of the sources instead of csrc/."""
    build_dir = out_dir or BUILD
    lib = os.path.join(build_dir, "libfa8.so")
    if not force and not ptxas_verbose and not defines and out_dir is None and src_dir is None and up_to_date():
        return LIB
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    srcs = sorted(glob.glob(os.path.join(src_dir, "*.cu"))) if src_dir else _sources()
    objs = [os.path.join(build_dir, os.path.basename(s)[:-3] + ".o") for s in srcs]

    def one(pair):
        src, obj = pair
        cmd = [cc, "-c", src, "-o", obj] + _flags(ptxas_verbose) + [f"-D{d}" for d in defines]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, r.returncode, r.stdout + r.stderr

    jobs = jobs or min(len(srcs), os.cpu_count() or 4)
    logs = []
    with cf.ThreadPoolExecutor(jobs) as ex:
        for src, rc, out in ex.map(one, zip(srcs, objs)):
            logs.append(f"== {os.path.basename(src)}\n{out}")
            if rc != 0:
                raise RuntimeError(f"nvcc failed on {src}:\n{out}")
    with open(os.path.join(build_dir, "ptxas.log"), "w") as f:
        f.write("\n".join(logs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, "-shared", "-o", tmp] + objs + ARCH + ["-Xcompiler", "-fPIC"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, ptxas_verbose="-v" in sys.argv))
