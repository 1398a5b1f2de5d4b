"""Build ``libfmha_gb300.so`` (and its checked twin) in-tree for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled by nvcc in parallel
(``-gencode arch=compute_103a,code=sm_103a -lineinfo -O3``) and linked into one
shared library next to this file.  The checked build compiles the same sources
with ``-DFMHA_CHECKED`` (every computed index of the kernels is tested before
its access, see ``include/fmha.h``) into ``libfmha_gb300_checked.so``.  Usage:
``python -m head_attention_forward_fmha_gb300.build [--force] [--verbose]
[--checked | --all]``.
"""
import argparse
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libfmha_gb300.so")
CHECKED_LIB_PATH = os.path.join(PKG, "libfmha_gb300_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def _variant(checked):
    """(library path, object directory, extra nvcc flags) of one build variant."""
    if checked:
        return CHECKED_LIB_PATH, BUILD_DIR + "_checked", ["-DFMHA_CHECKED"]
    return LIB_PATH, BUILD_DIR, []


def up_to_date(checked=False):
    lib = _variant(checked)[0]
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _build_variants(variants, force, verbose, extra_flags):
    todo = [c for c in variants if force or not up_to_date(c)]
    if not todo:
        return
    nvcc = _nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                     "--expt-relaxed-constexpr"] + list(extra_flags)
    if verbose:
        common += ["-Xptxas", "-v"]
    jobs = []
    for checked in todo:
        _, obj_dir, flags = _variant(checked)
        os.makedirs(obj_dir, exist_ok=True)
        for src in _sources():
            obj = os.path.join(obj_dir, os.path.splitext(os.path.basename(src))[0] + ".o")
            jobs.append((checked, src, obj, [nvcc] + common + flags + ["-c", src, "-o", obj]))

    def compile_one(job):
        r = subprocess.run(job[3], stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        return job, r.returncode, r.stdout

    objs = {c: [] for c in todo}
    with cf.ThreadPoolExecutor(max_workers=max(1, min(16, os.cpu_count() or 1))) as ex:
        for (checked, src, obj, _), rc, out in ex.map(compile_one, jobs):
            if rc != 0:
                raise RuntimeError("nvcc failed on %s%s:\n%s" % (src, " (checked)" if checked else "", out))
            if verbose and out.strip():
                sys.stdout.write(out)
            objs[checked].append(obj)
    for checked in todo:
        lib = _variant(checked)[0]
        tmp = lib + ".tmp"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs[checked] + ["-lcudart_static", "-ldl", "-lpthread", "-lrt"]
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s" % r.stdout)
        os.replace(tmp, lib)


def build(force=False, verbose=False, extra_flags=(), checked=False):
    """Build one variant (the normal library, or the checked one); returns its path."""
    _build_variants([checked], force, verbose, extra_flags)
    return _variant(checked)[0]


def build_all(force=False, verbose=False):
    """Build the normal and the checked library (all translation units in one pool)."""
    _build_variants([False, True], force, verbose, ())
    return LIB_PATH, CHECKED_LIB_PATH


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    g = ap.add_mutually_exclusive_group()
    g.add_argument("--checked", action="store_true", help="build only the checked library")
    g.add_argument("--all", action="store_true", help="build the normal and the checked library")
    args = ap.parse_args()
    if args.all:
        print("\n".join(build_all(force=args.force, verbose=args.verbose)))
    else:
        print(build(force=args.force, verbose=args.verbose, checked=args.checked))
