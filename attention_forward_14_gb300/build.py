"""Build libattn_fwd.so (sm_103a) in-tree with nvcc, and its checked variant.

Each translation unit under csrc/ is compiled in parallel, then linked into
``attention_forward_14_gb300/libattn_fwd.so``.  The checked variant,
``libattn_fwd_checked.so``, compiles every translation unit again with
ATTN_CHECKED=1 (every computed copy coordinate, output offset, decoded unit
and on-chip address of the forward and backward kernels is compared with
its bounds; a violation is recorded in the status word and the CTA winds
down).  Usage:
``python -m attention_forward_14_gb300.build [--force] [-v]``.
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libattn_fwd.so")
LIB_CHECKED = os.path.join(HERE, "libattn_fwd_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["attn_fwd_api.cu", "inst_d64.cu", "inst_d128_noncausal.cu", "inst_d128_causal.cu", "inst_fp8.cu",
           "attn_bwd_inst.cu", "attn_bwd_inst_varlen.cu"]
# the translation units compiled again, checked (all of them: forward and backward)
CHECKED_SOURCES = SOURCES


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "attn_fwd.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, checked: bool = True) -> str:
    """Build the library (and, with ``checked``, its checked variant) when a
    source is newer than it; returns the library's path."""
    deps = _deps()
    want = [(LIB, False)] + ([(LIB_CHECKED, True)] if checked else [])
    todo = [(lib, chk) for lib, chk in want if force or _stale(lib, deps)]
    if not todo:
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                    "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    if verbose:
        flags += ["-Xptxas", "-v"]

    def obj_path(src, chk):
        return os.path.join(BUILD, os.path.splitext(src)[0] + ("_checked.o" if chk else ".o"))

    def compile_one(job):
        src, chk = job
        obj = obj_path(src, chk)
        cmd = [cc, *flags, *(["-DATTN_CHECKED=1"] if chk else []), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}{' (checked)' if chk else ''}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    jobs = [(src, False) for src in SOURCES]
    jobs += [(src, True) for src in CHECKED_SOURCES if any(chk for _, chk in todo)]
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        list(ex.map(compile_one, jobs))
    for lib, chk in todo:
        objs = [obj_path(src, chk and src in CHECKED_SOURCES) for src in SOURCES]
        tmp = lib + f".tmp{os.getpid()}"
        r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose))


if __name__ == "__main__":
    main()
