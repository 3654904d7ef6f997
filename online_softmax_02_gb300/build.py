"""Build libattn.so in-tree with nvcc for sm_103a (no cmake, no torch
extension machinery): each .cu under csrc/ compiles to an object in
_build/ in parallel, then nvcc links the shared library next to this file.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build", "attn")
LIB = os.path.join(PKG, "libattn.so")
SOURCES = ["attn_api.cu", "fwd_sm103.cu", "bwd_sm103.cu", "fwd_f32.cu", "decode.cu", "softmax.cu"]
HEADERS = ["common.cuh", "ptx.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
                     "-Xcompiler", "-fPIC,-fvisibility=hidden",
                     "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn.so")
    return path


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), out: str | None = None,
          build_dir: str | None = None) -> str:
    """Compile (if needed) and return the path of libattn.so.

    ``extra_flags`` are added to every nvcc compile; a build with compile-time
    options other than the defaults goes to its own ``out`` library and
    ``build_dir`` (the default build stays untouched)."""
    LIB_OUT = LIB if out is None else out
    BUILD_DIR = BUILD if build_dir is None else build_dir
    os.makedirs(BUILD_DIR, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "attn.h")]
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [s, *hdrs]):
            cmd = [nvcc(), *NVCC_FLAGS, *extra_flags, "-c", s, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n%s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
        return r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(jobs) or 1) as ex:
        for out in ex.map(run, jobs):
            if verbose and out:
                print(out)
    if force or jobs or _stale(LIB_OUT, objs):
        tmp = LIB_OUT + ".tmp%d" % os.getpid()
        run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lrt",
             "-lpthread"])
        os.replace(tmp, LIB_OUT)
    return LIB_OUT


if __name__ == "__main__":
    # python -m online_softmax_02_gb300.build [--force] [-v] [-D NAME=VALUE ... --out PATH]
    # A build with -D options goes to its own library (--out) and build folder.
    import argparse
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", dest="verbose", action="store_true")
    ap.add_argument("-D", dest="defines", action="append", default=[],
                    help="compile-time option, e.g. -D ATTN_FWD_PAIR=1")
    ap.add_argument("--out", default=None, help="library path of a build with -D options")
    args = ap.parse_args()
    if args.defines and not args.out:
        ap.error("a build with -D options needs --out (the default library stays untouched)")
    out = os.path.abspath(args.out) if args.out else None
    bdir = None if out is None else os.path.join(os.path.dirname(out), "_objs")
    print(build(force=args.force, verbose=args.verbose,
                extra_flags=tuple("-D" + d for d in args.defines), out=out, build_dir=bdir))
