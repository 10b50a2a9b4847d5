"""Build the CUDA libraries in-tree with nvcc for sm_103a (B300).

  libedge0_moe.so   the layer library (csrc/*.cu), next to this file
  synth/_synth_fill.so   the device-side input generator used by tests and bench

Objects go to <repo>/_build/.  Rebuilds only what changed (source or header newer).
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
BUILD = os.path.join(ROOT, "_build")
NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr"]


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _run(cmds):
    procs = [(c, subprocess.Popen(c, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True))
             for c in cmds]
    failed = []
    for c, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((c, out))
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + out for c, out in failed)
        raise RuntimeError("nvcc failed:\n" + msg)


def _build_lib(sources, headers, out_so, extra_link=()):
    os.makedirs(BUILD, exist_ok=True)
    objs, cmds = [], []
    for src in sources:
        obj = os.path.join(BUILD, os.path.basename(os.path.dirname(src)) + "_" +
                           os.path.basename(src).replace(".cu", ".o"))
        objs.append(obj)
        if _newer(obj, [src] + headers):
            cmds.append([NVCC] + ARCH + FLAGS + ["-c", src, "-o", obj])
    _run(cmds)
    if cmds or _newer(out_so, objs):
        _run([[NVCC] + ARCH + ["-shared", "-cudart", "shared", "-o", out_so] + objs + list(extra_link)])
    return out_so


def build(verbose: bool = False) -> list[str]:
    csrc = os.path.join(PKG, "csrc")
    headers = glob.glob(os.path.join(csrc, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    libs = [_build_lib(sorted(glob.glob(os.path.join(csrc, "*.cu"))), headers,
                       os.path.join(PKG, "libedge0_moe.so"))]
    synth_dir = os.path.join(ROOT, "synth")
    libs.append(_build_lib([os.path.join(synth_dir, "fill.cu")], [],
                           os.path.join(synth_dir, "_synth_fill.so")))
    if verbose:
        print("built:", *libs)
    return libs


if __name__ == "__main__":
    build(verbose=True)
    sys.exit(0)
