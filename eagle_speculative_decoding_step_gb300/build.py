"""Builds libeaglespec.so in-tree with nvcc for sm_103a.

Each .cu translation unit compiles in parallel to an object file, then one
link step makes the shared library next to this file.  ``python -m
eagle_speculative_decoding_step_gb300.build`` runs it.

``build(timeline=True)`` (``-t`` on the command line) makes a second library,
libeaglespec_timeline.so, compiled with SPEC_TIMELINE: every kernel's first
thread records its block's start and end times into a log (see ``timeline.py``);
the product library has none of it.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libeaglespec.so")
BUILD = os.path.join(HERE, "_build")
OUT_TL = os.path.join(HERE, "libeaglespec_timeline.so")
BUILD_TL = os.path.join(HERE, "_build_timeline")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-v"]


def nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def build(verbose=False, force=False, timeline=False):
    out, bdir = (OUT_TL, BUILD_TL) if timeline else (OUT, BUILD)
    flags = FLAGS + (["-DSPEC_TIMELINE"] if timeline else [])
    srcs = sources()
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(os.path.dirname(HERE), "include", "eaglespec.h"))
    if not force and os.path.exists(out):
        t = os.path.getmtime(out)
        if all(os.path.getmtime(d) <= t for d in deps):
            return out
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()

    def comp(src):
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s%s" % (src, r.stdout, r.stderr))
        return obj, r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        res = list(ex.map(comp, srcs))
    objs = [o for o, _ in res]
    if verbose:
        for _, log in res:
            sys.stdout.write(log)
    tmp = out + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, timeline="-t" in sys.argv))
