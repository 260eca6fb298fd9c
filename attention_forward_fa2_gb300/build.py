"""Build the CUDA library in-tree: attention_forward_fa2_gb300/libfa_gb300.so.

nvcc compiles each translation unit for sm_103a in parallel, then links a
shared library with the C ABI of include/fa.h.  Usage:

    python -m attention_forward_fa2_gb300.build [--force] [--verbose] [--phase]
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa_gb300.so")
# The same sources with the phase clocks compiled in (FA_PHASE_CLOCKS=1).
BUILD_PHASE = os.path.join(PKG, "_build_phase")
LIB_PHASE = os.path.join(PKG, "libfa_gb300_phase.so")
UNITS = ("fa_api.cu", "fa_fwd_d128.cu", "fa_fwd_d128_bc64.cu", "fa_fwd_d128_causal.cu",
         "fa_fwd_d64.cu", "fa_fwd_d64_bc64.cu", "fa_fwd_d64_causal.cu", "fa_fwd_quad.cu",
         "fa_fwd_split.cu", "fa_static_scratch.cu", "fa_bwd.cu", "fa_fp8.cu",
         "fa_fp8_varlen.cu")
HEADERS = ("ptx.cuh", "fa_fwd_kernel.cuh", "fa_launch.h", "fa_combine.cuh", "fa_bwd_kernel.cuh")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC",
    "-Xptxas", "-v",
]


def nvcc() -> str:
    path = shutil.which("nvcc")
    if path:
        return path
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa_gb300.so")


def _newest_input() -> float:
    files = [os.path.join(CSRC, f) for f in UNITS + HEADERS]
    files.append(os.path.join(INCLUDE, "fa.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, phase: bool = False) -> str:
    """Compile (if stale) and return the path of the shared library.

    phase=True builds libfa_gb300_phase.so instead: the same sources with the
    kernel's phase clocks compiled in (fa_set_phase_buffer), for profiling."""
    lib, bdir = (LIB_PHASE, BUILD_PHASE) if phase else (LIB, BUILD)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input():
        return lib
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    defs = ["-DFA_PHASE_CLOCKS=1"] if phase else []
    procs = []
    for unit in UNITS:
        obj = os.path.join(bdir, unit.replace(".cu", ".o"))
        log = open(os.path.join(bdir, unit.replace(".cu", ".ptxas.log")), "w")
        cmd = [cc] + NVCC_FLAGS + defs + ["-I", INCLUDE, "-I", CSRC, "-c", os.path.join(CSRC, unit), "-o", obj]
        procs.append((unit, obj, log, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT)))
    failed = []
    for unit, obj, log, proc in procs:
        rc = proc.wait()
        log.close()
        if rc != 0:
            failed.append(unit)
        if verbose or rc != 0:
            with open(log.name) as f:
                sys.stderr.write(f.read())
    if failed:
        raise RuntimeError("nvcc failed for: %s" % ", ".join(failed))
    tmp = lib + ".tmp.%d" % os.getpid()
    link = [cc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp]
    link += [obj for _, obj, _, _ in procs]
    subprocess.run(link, check=True)
    os.replace(tmp, lib)
    return lib


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--phase", action="store_true", help="build libfa_gb300_phase.so (phase clocks)")
    args = ap.parse_args(argv)
    print(build(force=args.force, verbose=args.verbose, phase=args.phase))


if __name__ == "__main__":
    main()
