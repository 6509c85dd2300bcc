"""Build libfa.so in-tree: nvcc for sm_103a only, one object per source file,
compiled in parallel, linked with the static CUDA runtime.

    python -m causal_flash_attention_gb300.build            # libfa.so
    python -m causal_flash_attention_gb300.build --all      # + libfa_waittest.so

Variants (the same sources with one extra define each, never loaded by the
product path):
  trace     libfa_trace.so: kernels record per-role timelines into a buffer
            set with its extra export fa_trace_set(void*) (FA_TRACE).
  waittest  libfa_waittest.so: the bounded-wait limit shortened to about a
            millisecond and every tensor-core kernel made to wait first for a
            barrier phase that nothing completes (FA_WAIT_TEST), so that a test
            can check that a wait which runs out ends the kernel with an error
            status instead of a hang.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfa.so")
SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_fwd_pair.cu", "fa_bwd.cu", "fa_simt.cu", "fa_noalloc.cu",
           "fa_decode.cu"]
HEADERS = ["ptx.cuh", "fa_internal.h", "fa_decode.h", os.path.join("..", "..", "include", "fa.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "--expt-relaxed-constexpr"]
# ~1 ms at the GB300's SM clock
WAIT_TEST_LIMIT_CYCLES = 2_000_000
VARIANTS = {
    "": [],
    "trace": ["-DFA_TRACE"],
    "waittest": ["-DFA_WAIT_TEST", f"-DFA_WAIT_LIMIT_CYCLES={WAIT_TEST_LIMIT_CYCLES}LL"],
}


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def lib_path(variant: str = "") -> str:
    return LIB if not variant else LIB.replace("libfa.so", f"libfa_{variant}.so")


def _paths(variant: str):
    bdir = BUILD + (f"_{variant}" if variant else "")
    return bdir, lib_path(variant)


def build_variants(variants, verbose: bool = False, force: bool = False,
                   ptxas_verbose: bool = False) -> list:
    """Compile every stale object of the given variants in one parallel pool,
    then link each library; returns the library paths. Raises on errors."""
    cc = nvcc()
    headers = [os.path.join(CSRC, h) for h in HEADERS]
    jobs = []
    for variant in variants:
        bdir, _ = _paths(variant)
        os.makedirs(bdir, exist_ok=True)
        for src in SOURCES:
            s = os.path.join(CSRC, src)
            o = os.path.join(bdir, src.replace(".cu", ".o"))
            if force or _stale(o, [s] + headers):
                cmd = [cc, *ARCH, *CFLAGS, *VARIANTS[variant], "-c", s, "-o", o]
                if ptxas_verbose:
                    cmd += ["-Xptxas", "-v"]
                jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with concurrent.futures.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), 32))) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or ptxas_verbose or r.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {cmd[-3]}")
    libs = []
    for variant in variants:
        bdir, lib = _paths(variant)
        objs = [os.path.join(bdir, s.replace(".cu", ".o")) for s in SOURCES]
        if force or _stale(lib, objs):
            tmp = lib + ".tmp"
            cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-ldl", "-lrt",
                   "-lpthread"]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if verbose or r.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"link of {os.path.basename(lib)} failed")
            os.replace(tmp, lib)
        libs.append(lib)
    return libs


def build(verbose: bool = False, force: bool = False, ptxas_verbose: bool = False,
          trace: bool = False, variant: str = "") -> str:
    """Compile and link libfa.so (or the named variant); returns its path."""
    v = "trace" if trace else variant
    return build_variants([v], verbose, force, ptxas_verbose)[0]


def build_all(verbose: bool = False, force: bool = False) -> list:
    """The product library and the wait-limit test library, compiled together."""
    return build_variants(["", "waittest"], verbose, force)


if __name__ == "__main__":
    if "--all" in sys.argv:
        print(build_all(verbose=True, force="--force" in sys.argv))
    else:
        print(build(verbose=True, force="--force" in sys.argv, ptxas_verbose="-v" in sys.argv,
                    trace="--trace" in sys.argv))
