"""Builds libdt.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into one shared
library next to this file. ``python -m dynamic_draft_tree_gb300.build``.
"""
import os
import platform
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libdt.so")
ARCH = "103a"

SOURCES = ["dt_api.cu", "k_tree.cu", "k_select.cu", "k_meta.cu", "k_verify.cu", "k_graft.cu",
           "k_rowtopk_static.cu", "k_kv.cu", "k_block.cu", "k_sampled.cu"]
HEADERS = ["dt_internal.cuh", "rowscan.cuh", "rowstream.cuh", "cast_block.cuh"]


def nvcc_flags(verbose_ptxas=False):
    f = ["-O3", "-std=c++17", f"-gencode=arch=compute_{ARCH},code=sm_{ARCH}", "-lineinfo",
         "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


_ELF_MACHINE = {"x86_64": 62, "aarch64": 183, "arm64": 183}


def elf_matches_host(path):
    """True if the ELF file at path was built for this machine's architecture."""
    want = _ELF_MACHINE.get(platform.machine())
    try:
        with open(path, "rb") as f:
            head = f.read(20)
    except OSError:
        return False
    if len(head) < 20 or head[:4] != b"\x7fELF" or want is None:
        return False
    return int.from_bytes(head[18:20], "little") == want


def _stale(out, deps):
    if not os.path.exists(out) or not elf_matches_host(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose_ptxas=False, quiet=True):
    os.makedirs(BUILD, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "dt.h")]
    procs, objs = [], []
    for src in SOURCES:
        sp = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or verbose_ptxas or _stale(obj, [sp] + hdrs):
            cmd = ["nvcc", *nvcc_flags(verbose_ptxas), "-c", sp, "-o", obj]
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif text.strip() and (verbose_ptxas or not quiet):
            print(f"--- {src}\n{text}")
    if failed:
        msg = "\n".join(f"--- {s}\n{t}" for s, t in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    if force or _stale(LIB, objs):
        subprocess.check_call(["nvcc", "-shared", f"-gencode=arch=compute_{ARCH},code=sm_{ARCH}",
                               "-o", LIB, *objs, "-lcudart"])
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, quiet=False)
    print(LIB)
