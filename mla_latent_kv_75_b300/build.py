"""Build libmla.so in-tree from the CUDA sources in csrc/ (sm_103a only).

Each .cu file is compiled separately with relocatable device code, then device-linked into
one shared library next to this file. Run ``python mla_latent_kv_75_b300/build.py``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libmla.so")
BUILD = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-rdc=true", "-Xcompiler", "-fPIC",
         "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths.append(os.path.join(ROOT, "include", "mla.h"))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    """Compile every csrc/*.cu for sm_103a and link libmla.so; returns its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-rdc=true", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    _write_build_info()
    return LIB


def _write_build_info() -> None:
    """Record the commit the library was built from, for a copy of the tree that runs
    without its .git directory; reporting only."""
    import json
    info = {"git": None, "dirty": None}
    try:
        sha = subprocess.run(["git", "-C", ROOT, "rev-parse", "HEAD"], capture_output=True,
                             text=True, timeout=10)
        st = subprocess.run(["git", "-C", ROOT, "status", "--porcelain", "--", "mla_latent_kv_75_b300",
                             "include"], capture_output=True, text=True, timeout=10)
        if sha.returncode == 0:
            info = {"git": sha.stdout.strip(), "dirty": bool(st.stdout.strip())}
    except Exception:
        pass
    path = os.path.join(BUILD, "build_info.json")
    if info["git"] is None and os.path.exists(path):
        # a tree without git (a copy of a built checkout): keep the commit recorded by the
        # build it was copied from; the bench's source hash tells whether the sources match
        try:
            prev = json.load(open(path))
            if prev.get("git"):
                info = {"git": prev["git"], "dirty": prev.get("dirty"), "rebuilt_without_git": True}
        except Exception:
            pass
    with open(path, "w") as f:
        json.dump(info, f)


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else []
    print(build(force=True, verbose=v or bool(extra), extra=extra))
