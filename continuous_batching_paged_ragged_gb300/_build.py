"""Build libpkv.so (the C-ABI library) and libpkv_synth.so (the device input generator) in-tree with nvcc.

Objects go to ``_build/`` at the repository root; the shared libraries land next to this file.  Translation
units compile in parallel; a library is rebuilt only when a source or header is newer than it.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from typing import List

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]

LIBS = {
    "libpkv.so": ["pool.cu", "attention.cu", "decode_e4m3.cu", "prefill.cu", "sched.cpp"],
    "libpkv_synth.so": ["synth.cu"],
}


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _headers() -> List[str]:
    hs = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    hs += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return hs


def _stale(target: str, deps: List[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, extra_flags: List[str] = ()) -> List[str]:
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    headers = _headers()
    jobs = []
    plan = []
    for lib, srcs in LIBS.items():
        objs = []
        for src in srcs:
            s = os.path.join(CSRC, src)
            o = os.path.join(BUILD, src + ".o")
            objs.append(o)
            if force or _stale(o, [s] + headers):
                cmd = [nvcc] + ARCH + NVCC_FLAGS + list(extra_flags) + ["-c", s, "-o", o]
                if src.endswith(".cpp"):
                    cmd = [nvcc] + NVCC_FLAGS + ["-x", "c++", "-c", s, "-o", o]
                if verbose:
                    print(" ".join(cmd), flush=True)
                jobs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        plan.append((lib, objs))
    failed = []
    for src, p in jobs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append(f"--- {src} ---\n{text}")
        elif verbose and text.strip():
            print(text, flush=True)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    built = []
    for lib, objs in plan:
        target = os.path.join(PKG, lib)
        if force or _stale(target, objs):
            cmd = [nvcc] + ARCH + ["-shared", "-o", target] + objs + ["-lcudart"]
            if verbose:
                print(" ".join(cmd), flush=True)
            r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
            if r.returncode != 0:
                raise RuntimeError(f"link of {lib} failed:\n{r.stdout.decode(errors='replace')}")
        built.append(target)
    return built


if __name__ == "__main__":
    for path in build(verbose="-v" in sys.argv, force="-f" in sys.argv):
        print(path)
