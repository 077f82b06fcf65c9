"""Builds the C-ABI library ``libdlo.so`` from ``csrc/`` with nvcc for sm_103a.

Each translation unit compiles in its own process (in parallel) into
``_build/``, then nvcc links the shared library into the package directory.
Rebuilds only what changed (source newer than object, or a header newer).
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libdlo.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))


def _compile(src, nvcc, newest_header, extra):
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), newest_header):
        return obj, None
    cmd = [nvcc] + ARCH + NVCC_FLAGS + extra + ["-c", src, "-o", obj + ".tmp"]
    if src.endswith(".cpp"):
        cmd = [nvcc] + NVCC_FLAGS + extra + ["-x", "c++", "-c", src, "-o", obj + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        return obj, "compile failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr)
    os.replace(obj + ".tmp", obj)
    return obj, r.stderr if "warning" in r.stderr.lower() else None


def build(verbose=False, ptxas_info=False, force=False):
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    newest = max(os.path.getmtime(h) for h in _headers())
    if force:
        newest = float("inf")
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    objs, errs = [], []
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        for obj, msg in ex.map(lambda s: _compile(s, nvcc, newest, extra), srcs):
            objs.append(obj)
            if msg:
                (errs if msg.startswith("compile failed") else [None]).append(msg)
                if verbose or ptxas_info:
                    sys.stderr.write(msg + "\n")
    errs = [e for e in errs if e]
    if errs:
        raise RuntimeError("\n".join(errs))
    if (not os.path.exists(LIB) or force
            or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs)):
        tmp = LIB + ".tmp%d" % os.getpid()
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs + ["-ldl"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed: %s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv, force="--force" in sys.argv))
