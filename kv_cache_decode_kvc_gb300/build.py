"""Builds libkvc.so (the CUDA library behind include/kvc.h) for sm_103a with nvcc.

Every translation unit compiles in parallel into ``_build/``; the decode kernel's TU is
compiled once per (dtype, head dim).  The shared library links the CUDA runtime statically,
so loading it needs no GPU.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libkvc.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]

# (object name, source, extra defines)
DECODE_INST = [("bf16", 64), ("bf16", 128), ("bf16", 256),
               ("f32", 4), ("f32", 64), ("f32", 128), ("f32", 256)]


def _units():
    units = [("kvc_host", "kvc_host.cu", []), ("kvc_copy", "kvc_copy.cu", []),
             ("kvc_noalloc", "kvc_noalloc.cu", []), ("kvc_selftest", "kvc_selftest.cu", [])]
    for d in (64, 128, 256):
        units.append((f"kvc_decode_tc_d{d}", "kvc_decode_tc_inst.cu", [f"-DKVC_INST_D={d}"]))
    units.append(("kvc_decode_tc5_d128", "kvc_decode_tc5_inst.cu", ["-DKVC_TC5_MODE=0"]))
    units.append(("kvc_decode_tc5p_d128", "kvc_decode_tc5_inst.cu", ["-DKVC_TC5_MODE=1"]))
    units.append(("kvc_decode_tc5r_d128", "kvc_decode_tc5_inst.cu", ["-DKVC_TC5_MODE=2"]))
    units.append(("kvc_decode_tc5q_d128", "kvc_decode_tc5_inst.cu", ["-DKVC_TC5_MODE=3"]))
    units.append(("kvc_decode_tc5f_d128", "kvc_decode_tc5_inst.cu", ["-DKVC_TC5_MODE=4"]))
    for dt, d in DECODE_INST:
        units.append((f"kvc_decode_{dt}_d{d}", "kvc_decode_inst.cu",
                      [f"-DKVC_INST_BF16={1 if dt == 'bf16' else 0}", f"-DKVC_INST_D={d}"]))
    return units


def _sources():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(os.path.dirname(PKG), "include", "kvc.h")]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, jobs: int | None = None) -> str:
    os.makedirs(BUILD, exist_ok=True)
    deps = _sources()
    units = _units()
    objs = []
    todo = []
    for name, src, defs in units:
        obj = os.path.join(BUILD, name + ".o")
        objs.append(obj)
        if force or _stale(obj, deps):
            cmd = ["nvcc", *ARCH, *FLAGS, *defs, "-c", os.path.join(CSRC, src), "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            todo.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    if todo:
        with cf.ThreadPoolExecutor(max_workers=jobs or min(len(todo), os.cpu_count() or 4)) as ex:
            for cmd, r in ex.map(run, todo):
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
                if verbose:
                    sys.stderr.write(r.stderr)
    if force or todo or _stale(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = ["nvcc", *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
