"""Test helpers for the library's NVTX ranges: build the recording NVTX
tool (tests/nvtx_probe.c) with the host C compiler, run a Python snippet in
a fresh process with the tool attached through NVTX_INJECTION64_PATH, and
read back what it recorded (no method arithmetic here)."""
import ctypes
import json
import os
import shutil
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROBE_SRC = os.path.join(ROOT, "tests", "nvtx_probe.c")


def cuda_include():
    for nvcc in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if nvcc and os.path.exists(nvcc):
            inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))),
                               "include")
            if os.path.exists(os.path.join(inc, "nvtx3", "nvToolsExt.h")):
                return inc
    raise RuntimeError("no CUDA include directory with nvtx3 found")


def build_probe(out_dir):
    """Compiles the tool into out_dir and returns its path."""
    so = os.path.join(str(out_dir), "libnvtx_probe.so")
    cc = shutil.which("gcc") or shutil.which("cc")
    cmd = [cc, "-shared", "-fPIC", "-O2", "-I", cuda_include(), "-o", so, PROBE_SRC,
           "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("probe build failed: %s\n%s" % (" ".join(cmd), r.stderr))
    return so


def read_probe(path):
    """The events the tool recorded in this process, as dicts, in order."""
    L = ctypes.CDLL(path)
    L.probe_count.restype = ctypes.c_int64
    L.probe_dropped.restype = ctypes.c_int64
    L.probe_inits.restype = ctypes.c_int32
    L.probe_event_at.restype = ctypes.c_int32
    L.probe_event_at.argtypes = [ctypes.c_int64] + [ctypes.c_void_p] * 6
    kind, depth = ctypes.c_int32(), ctypes.c_int32()
    payload, thread = ctypes.c_int64(), ctypes.c_uint64()
    name, domain = ctypes.create_string_buffer(48), ctypes.create_string_buffer(48)
    out = []
    for i in range(L.probe_count()):
        ok = L.probe_event_at(i, ctypes.byref(kind), ctypes.byref(depth), ctypes.byref(payload),
                              ctypes.byref(thread), name, domain)
        assert ok
        out.append({"kind": "push" if kind.value == 1 else "pop", "depth": depth.value,
                    "payload": payload.value, "thread": thread.value,
                    "name": name.value.decode(), "domain": domain.value.decode()})
    return {"events": out, "dropped": L.probe_dropped(), "inits": L.probe_inits()}


def run_traced(snippet, probe, timeout=600):
    """Runs `snippet` (Python source that sets a JSON-serialisable `result`)
    in a fresh interpreter with the tool attached; returns (result, probe
    record)."""
    code = ("import json, sys\nsys.path.insert(0, %r)\n" % ROOT + snippet +
            "\nfrom tests._nvtx import read_probe\n"
            "print('@@' + json.dumps({'result': result, 'probe': read_probe(%r)}))\n" % probe)
    env = dict(os.environ, NVTX_INJECTION64_PATH=probe)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       cwd=ROOT, timeout=timeout)
    if r.returncode != 0:
        raise RuntimeError("traced run failed (%d):\n%s\n%s" % (r.returncode, r.stdout[-4000:],
                                                              r.stderr[-4000:]))
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("@@")][-1]
    d = json.loads(line[2:])
    return d["result"], d["probe"]


def ranges(events, domain="dlo"):
    """Matched (name, payload, depth, thread) of every push in `domain`, in
    push order, with a check that each thread's pushes and pops pair up."""
    stacks, out = {}, []
    for e in events:
        st = stacks.setdefault(e["thread"], [])
        if e["kind"] == "push":
            assert e["depth"] == len(st), e
            st.append(e)
            if e["domain"] == domain:
                out.append((e["name"], e["payload"], e["depth"], e["thread"]))
        else:
            assert st, "pop with no open range: %r" % (e,)
            st.pop()
            assert e["depth"] == len(st), e
    for t, st in stacks.items():
        assert not st, "ranges left open on thread %d: %r" % (t, st)
    return out
