"""Builds the paged-KV CUDA library in-tree with nvcc for sm_103a.

    python -m paged_kv_cache_217_gb300.build [--force] [--verbose]

Objects go to ``paged_kv_cache_217_gb300/_build/`` and the shared library to
``paged_kv_cache_217_gb300/_lib/libpaged_kv.so`` (both git-ignored). Translation
units compile in parallel; a unit is rebuilt when it or any header in
``csrc/`` or ``include/`` is newer than its object.
"""

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
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "libpaged_kv.so")

SOURCES = [
    "api.cu",
    "decode_noalloc.cu",
    "decode_f16.cu",
    "decode_bf16.cu",
    "decode_int8.cu",
    "cache_ops.cu",
    "diag.cu",
    "block_manager.cpp",
    "status.cpp",
]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put CUDA 13 on PATH)")


def _headers():
    out = []
    for d in (CSRC, INCLUDE):
        for f in os.listdir(d):
            if f.endswith((".h", ".cuh", ".hpp")):
                out.append(os.path.join(d, f))
    return out


def _cmd(nvcc, src, obj, ptxas_verbose, defines=()):
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC, "-Xcompiler", "-fPIC"] + \
        [f"-D{d}" for d in defines]
    if src.endswith(".cu"):
        extra = ARCH + ["-lineinfo", "--expt-relaxed-constexpr"]
        if ptxas_verbose:
            extra += ["-Xptxas", "-v"]
        return [nvcc] + common + extra + ["-c", src, "-o", obj]
    return [nvcc] + common + ["-x", "c++", "-c", src, "-o", obj]


def build(force=False, verbose=False, ptxas_verbose=False, defines=(), out_dir=None):
    """Compile every translation unit and link libpaged_kv.so; returns its path.

    ``defines`` (NAME=VALUE strings) and ``out_dir`` build a variant (the
    per-CTA tracing build, PKV_TRACE=1, or the CUDA-core INT8 tile,
    PKV_INT8_MMA=0) into a directory of its own instead of the package.
    """
    build_dir = os.path.join(out_dir, "_build") if out_dir else BUILD
    lib_path = os.path.join(out_dir, "libpaged_kv.so") if out_dir else LIB
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(os.path.dirname(lib_path), exist_ok=True)
    nvcc = _nvcc()
    newest_header = max((os.path.getmtime(h) for h in _headers()), default=0.0)
    procs, objs = [], []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(build_dir, s + ".o")
        objs.append(obj)
        stale = force or not os.path.exists(obj) or \
            os.path.getmtime(obj) < max(os.path.getmtime(src), newest_header)
        if stale:
            cmd = _cmd(nvcc, src, obj, ptxas_verbose, defines)
            if verbose:
                print(" ".join(cmd), flush=True)
            procs.append((s, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                              text=True)))
    failed = []
    for s, p in procs:
        out, _ = p.communicate()
        if out and (verbose or ptxas_verbose or p.returncode):
            print(out, end="", flush=True)
        if p.returncode:
            failed.append(s)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    if procs or force or not os.path.exists(lib_path) or \
            os.path.getmtime(lib_path) < max(os.path.getmtime(o) for o in objs):
        tmp = lib_path + ".tmp"
        cmd = [nvcc, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib_path)
    return lib_path


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    ap.add_argument("--define", action="append", default=[], help="NAME=VALUE passed to nvcc as -D")
    ap.add_argument("--out-dir", default=None, help="build a variant into this directory")
    args = ap.parse_args(argv)
    print(build(force=args.force, verbose=args.verbose, ptxas_verbose=args.ptxas_verbose,
                defines=args.define, out_dir=args.out_dir))


if __name__ == "__main__":
    sys.exit(main())
