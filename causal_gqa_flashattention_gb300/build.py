"""Build ``libnea_attn.so`` in-tree from ``csrc/*.cu`` for sm_103a.

Each translation unit is compiled by its own nvcc process (in parallel), then
linked into one shared library with the CUDA runtime linked statically, so the
library has no link-time dependency on libcudart or libcuda.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libnea_attn.so")
OBJDIR = os.path.join(HERE, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-diag-suppress", "177"]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hdrs.append(os.path.join(os.path.dirname(HERE), "include", "nea_attn.h"))
    return hdrs


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in sources() + _deps() + [__file__])


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(OBJDIR, exist_ok=True)
    procs = []
    for src in sources():
        obj = os.path.join(OBJDIR, os.path.basename(src)[:-3] + ".o")
        cmd = ["nvcc", *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((src, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                 stderr=subprocess.STDOUT, text=True)))
    objs, failed = [], []
    for src, obj, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stderr.write(out)
        if p.returncode != 0:
            failed.append(src)
        objs.append(obj)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run(["nvcc", *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB)
    return LIB


def build_variant(name: str, flags) -> str:
    """Build the library with extra nvcc flags into _build/<name>/ (a separate
    copy used by tests, e.g. the build whose bounded waits run out quickly);
    returns its path.  The default library is not touched."""
    global LIB, OBJDIR
    saved = LIB, OBJDIR
    try:
        OBJDIR = os.path.join(HERE, "_build", name)
        LIB = os.path.join(OBJDIR, "libnea_attn.so")
        return build(force=True, extra_flags=tuple(flags))
    finally:
        LIB, OBJDIR = saved


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
