"""Builds the CUDA library (libfa_fwd.so) in-tree for sm_103a with nvcc.

One object per translation unit, compiled in parallel, then linked against the
shared CUDA runtime so the library and PyTorch share one runtime instance.
"""
from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa_fwd.so")
TRACE_LIB = os.path.join(PKG, "libfa_fwd_trace.so")
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def is_stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs())


def variant_lib(trace: bool = False, exp2_poly_pairs: int = 0, epilogue_in_softmax: bool = False,
                debug_stats: bool = False, score_rotation: bool = False, pv_split: bool = False) -> str:
    """Path of the library built with these options."""
    if debug_stats:
        return os.path.join(PKG, "libfa_fwd_dbg.so")
    if exp2_poly_pairs or epilogue_in_softmax or score_rotation or pv_split:
        tag = (f"poly{exp2_poly_pairs}" if exp2_poly_pairs else "") + ("epism" if epilogue_in_softmax else "") + \
            ("rot" if score_rotation else "") + ("pvsplit" if pv_split else "")
        return os.path.join(PKG, f"libfa_fwd_{tag}.so")
    return TRACE_LIB if trace else LIB


def _compile(src: str, ptxas_verbose: bool, trace: bool = False, exp2_poly_pairs: int = 0,
             epilogue_in_softmax: bool = False, debug_stats: bool = False,
             score_rotation: bool = False, pv_split: bool = False) -> tuple[str, str]:
    tag = (".trace" if trace else "") + (f".poly{exp2_poly_pairs}" if exp2_poly_pairs else "") + \
        (".epism" if epilogue_in_softmax else "") + (".dbg" if debug_stats else "") + \
        (".rot" if score_rotation else "") + (".pvsplit" if pv_split else "")
    obj = os.path.join(OBJDIR, os.path.basename(src) + tag + ".o")
    cmd = [NVCC, *ARCH, *FLAGS, "-c", src, "-o", obj] + (["-DFA_TRACE"] if trace else [])
    if debug_stats:
        cmd.append("-DFA_DEBUG_STATS")
    if exp2_poly_pairs:
        cmd.append(f"-DFA_EXP2_POLY_PAIRS={exp2_poly_pairs}")
    if epilogue_in_softmax:
        cmd.append("-DFA_EPILOGUE_IN_SOFTMAX=1")
    if score_rotation:
        cmd.append("-DFA_SCORE_ROTATION=1")
    if pv_split:
        cmd.append("-DFA_PV_SPLIT=1")
    if ptxas_verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, ptxas_verbose: bool = False, jobs: int | None = None,
          trace: bool = False, exp2_poly_pairs: int = 0, epilogue_in_softmax: bool = False,
          debug_stats: bool = False, score_rotation: bool = False, pv_split: bool = False) -> str:
    """Compile every CUDA translation unit and link libfa_fwd.so (or, with
    trace=True, the event-tracing variant libfa_fwd_trace.so; with
    exp2_poly_pairs=N in 1..16, libfa_fwd_polyN.so, whose softmax computes N of
    every 16 exponential pairs on the FMA pipe; with epilogue_in_softmax,
    libfa_fwd_epism.so, whose softmax warpgroups also run the epilogue; with
    debug_stats, libfa_fwd_dbg.so, which writes each row's final base and sum
    and counts its re-bases; with score_rotation, libfa_fwd_rot.so, whose D=64
    kernels rotate three score buffers; with pv_split, libfa_fwd_pvsplit.so,
    whose softmax publishes P in two halves); returns its path."""
    if not 0 <= exp2_poly_pairs <= 16:
        raise ValueError("exp2_poly_pairs must be in [0, 16]")
    lib = variant_lib(trace, exp2_poly_pairs, epilogue_in_softmax, debug_stats, score_rotation, pv_split)
    if not force and not ptxas_verbose and not is_stale(lib):
        return lib
    os.makedirs(OBJDIR, exist_ok=True)
    srcs = sources()
    with ThreadPoolExecutor(max_workers=jobs or min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda s: _compile(s, ptxas_verbose, trace, exp2_poly_pairs, epilogue_in_softmax,
                                                 debug_stats, score_rotation, pv_split), srcs))
    if ptxas_verbose:
        for _, log in results:
            if log.strip():
                print(log)
    tmp = lib + ".tmp"
    cmd = [NVCC, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *[o for o, _ in results],
           "-Xlinker", f"-rpath,{os.path.join(CUDA_HOME, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def ptxas_report(jobs: int | None = None) -> list[dict]:
    """Compiles every translation unit with ``-Xptxas -v`` (objects in a
    scratch folder, the library untouched) and returns, per kernel instance,
    ptxas's register count at launch, stack frame and spill bytes."""
    import re
    import shutil
    import tempfile
    tmp = tempfile.mkdtemp(prefix="fa_ptxas_")
    try:
        def one(src):
            obj = os.path.join(tmp, os.path.basename(src) + ".o")
            cmd = [NVCC, *ARCH, *FLAGS, "-c", src, "-o", obj, "-Xptxas", "-v"]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
            return os.path.basename(src), r.stderr
        srcs = sources()
        with ThreadPoolExecutor(max_workers=jobs or min(len(srcs), os.cpu_count() or 4)) as ex:
            logs = list(ex.map(one, srcs))
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    rows = []
    for unit, log in logs:
        cur = None
        for line in log.splitlines():
            m = re.search(r"Compiling entry function '(\S+)'", line)
            if m:
                cur = {"unit": unit, "mangled": m.group(1)}
                continue
            m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads", line)
            if m and cur is not None:
                cur["stack"], cur["spill_stores"], cur["spill_loads"] = (int(x) for x in m.groups())
                continue
            m = re.search(r"Used (\d+) registers", line)
            if m and cur is not None:
                cur["registers"] = int(m.group(1))
                rows.append(cur)
                cur = None
    names = [r["mangled"] for r in rows]
    try:
        out = subprocess.run(["c++filt"], input="\n".join(names), capture_output=True, text=True,
                             check=True).stdout.splitlines()
    except (OSError, subprocess.CalledProcessError):
        out = names
    for r, n in zip(rows, out):
        r["kernel"] = n.replace("(anonymous namespace)::", "").split("(")[0]
    return rows


if __name__ == "__main__":
    import sys
    if "--ptxas-report" in sys.argv:
        print("| translation unit | kernel | registers at launch | stack bytes | spill stores | spill loads |")
        print("|---|---|---|---|---|---|")
        for r in sorted(ptxas_report(), key=lambda r: (r["unit"], r["kernel"])):
            print(f"| {r['unit']} | `{r['kernel']}` | {r['registers']} | {r['stack']} | {r['spill_stores']} | "
                  f"{r['spill_loads']} |")
    else:
        print(build(force=True, ptxas_verbose="-v" in sys.argv, trace="--trace" in sys.argv))
