"""Builds libverify.so (the C-ABI library) in-tree with nvcc for sm_103a.

Nine translation units are compiled in parallel (host API + packers, the streaming executor for
8/16 token columns, the executor for 24/32 token columns, the executor with the Q4 unit, the
sampled acceptance, the verify attention, the Gated DeltaNet scan, the decode loop, the error
bookkeeping) and linked against the shared CUDA runtime.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libverify.so")
# The same library with the executor's phase timeline recorded (trace.cuh): a measurement build.
BUILD_TRACE = os.path.join(PKG, "_build_trace")
LIB_TRACE = os.path.join(PKG, "libverify_trace.so")
# The same library with tiny limits on every bounded device wait and a workspace hook that makes
# one CTA skip its first grid-barrier arrival: the build in which a test makes a wait run out.
BUILD_WAIT = os.path.join(PKG, "_build_waittest")
LIB_WAIT = os.path.join(PKG, "libverify_waittest.so")
# A measurement build of the executor's unit loop alone (csrc/unit_bench.cu; unit_bench.py runs it).
BUILD_UNIT = os.path.join(PKG, "_build_unitbench")
LIB_UNIT = os.path.join(PKG, "libverify_unitbench.so")
VARIANTS = {"": (LIB, BUILD, []), "trace": (LIB_TRACE, BUILD_TRACE, ["-DVP_PHASE_TRACE"]),
            "waittest": (LIB_WAIT, BUILD_WAIT, ["-DVP_WAIT_TEST"]), "unitbench": (LIB_UNIT, BUILD_UNIT, [])}
UNIT_SOURCES = ["unit_bench.cu"]
SOURCES = ["api.cu", "exec_nt12.cu", "exec_nt34.cu", "exec_q4.cu", "sample.cu", "attention.cu", "gdn.cu",
           "loop.cu", "errors.cu", "mixer.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]


def _inputs():
    files = [os.path.join(INCLUDE, "verify.h")]
    for f in os.listdir(CSRC):
        files.append(os.path.join(CSRC, f))
    return files


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, trace: bool = False, variant: str = "") -> str:
    """Builds libverify.so (or a measurement / test variant of it: "trace" with the phase timeline,
    "waittest" with tiny wait limits, "unitbench" the unit-loop breakdown alone; trace=True is
    variant "trace") and returns its path; nothing is rebuilt when the library is newer than every
    source."""
    lib, bdir, defs = VARIANTS["trace" if trace else variant]
    deps = _inputs()
    if not force and not _stale(lib, deps):
        return lib
    os.makedirs(bdir, exist_ok=True)
    procs = []
    objs = []
    for src in UNIT_SOURCES if variant == "unitbench" else SOURCES:
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = ["nvcc", *ARCH, *FLAGS, *defs, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stderr.write(out)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.run(["nvcc", *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, trace="--trace" in sys.argv,
                variant="waittest" if "--waittest" in sys.argv else ""))
