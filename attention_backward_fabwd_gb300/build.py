"""Build libfabwd.so in-tree with nvcc for sm_103a (no cmake; translation units in parallel)."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libfabwd.so")

# (source, object, defines): the kernel families are compiled once per io dtype
_PLAIN = ["fabwd_api.cu", "fabwd_aux.cu", "fabwd_static_ws.cu"]
_PER_DTYPE = ["fabwd_onegrid.cu", "fabwd_split.cu", "fabwd_fused.cu", "fabwd_forward.cu"]
UNITS = [(src, src.replace(".cu", ".o"), []) for src in _PLAIN] + [
    (src, src.replace(".cu", f"_{dt}.o"), [f"-DFABWD_INST_FP16={int(dt == 'fp16')}"])
    for src in _PER_DTYPE for dt in ("bf16", "fp16")]
SOURCES = _PLAIN + _PER_DTYPE
HEADERS = ["fabwd_ptx.cuh", "fabwd_internal.cuh", "fabwd_main.cuh", "fabwd_dq.cuh", "fabwd_kv.cuh", "fabwd_sep.cuh", "fabwd_fwd.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "fabwd.h"), __file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile every translation unit for sm_103a and link libfabwd.so; returns its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(OUT, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for src, o, defines in UNITS:
        obj = os.path.join(OUT, o)
        objs.append(obj)
        cmd = [cc, *ARCH, *FLAGS, *defines, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    errors = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            errors.append(f"--- {src}\n{out}")
        elif verbose and out.strip():
            print(out, file=sys.stderr)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-ldl"]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
