"""Builds libpagedkv.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in its own nvcc process, in parallel; the decode
kernel is compiled once per (cache type, dtype, head_dim) and the multi-token
balanced kernel once per (cache type, dtype). The library links the CUDA
runtime statically and needs no libcuda at link time (the tensor-map encoder
is fetched through the runtime's driver entry-point query).

Usage: python -m paged_kv_cache_114_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libpagedkv.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-O3",
                "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _units():
    units = [("pa_api", "pa_api.cu", []), ("pa_cache_ops", "pa_cache_ops.cu", []),
             ("pa_decode_reduce", "pa_decode_reduce.cu", []),
             ("pa_noalloc", "pa_noalloc.cu", []), ("pa_prefill", "pa_prefill.cu", []),
             ("pa_prefix_hash", "pa_prefix_hash.cu", []),
             ("pa_prefill_tc", "pa_prefill_tc.cu", []),
             ("pa_prefill_tc128", "pa_prefill_tc128.cu", [])]
    for bf in (0, 1):
        for d in (64, 128, 256):
            tag = f"pa_decode_{'bf16' if bf else 'f16'}_{d}"
            units.append((tag, "pa_decode_inst.cu", [f"-DPA_INST_BF16={bf}", f"-DPA_INST_D={d}"]))
        for d in (128, 256):  # E4M3 caches
            tag = f"pa_decode_e4m3_{'bf16' if bf else 'f16'}_{d}"
            units.append((tag, "pa_decode_inst.cu", [f"-DPA_INST_BF16={bf}", f"-DPA_INST_D={d}",
                                                     "-DPA_INST_FP8=1"]))
        for fp8 in (0, 1):  # few new tokens per sequence on the grouped balanced kernel
            tag = f"pa_verify_{'e4m3_' if fp8 else ''}{'bf16' if bf else 'f16'}"
            units.append((tag, "pa_verify_inst.cu", [f"-DPA_INST_BF16={bf}", f"-DPA_INST_FP8={fp8}"]))
    return units


def _sources():
    out = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    out.append(os.path.join(ROOT, "include", "pa.h"))
    out.append(os.path.abspath(__file__))
    return out


def _nvcc():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedkv")
    return nvcc


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(s) <= t for s in _sources())


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    """Compile every CUDA translation unit and link libpagedkv.so; returns its path."""
    if not force and up_to_date():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = list(extra_flags or [])

    def compile_one(unit):
        tag, src, defs = unit
        obj = os.path.join(BUILD_DIR, tag + ".o")
        cmd = [nvcc, *ARCH_FLAGS, *COMMON_FLAGS, *extra, *defs, "-c", os.path.join(CSRC, src),
               "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {tag}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(f"[{tag}]\n{r.stdout}{r.stderr}")
        return obj

    workers = min(len(_units()), max(1, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        objs = list(ex.map(compile_one, _units()))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true", help="print ptxas resource usage")
    args = ap.parse_args(argv)
    extra = ["-Xptxas", "-v"] if args.verbose else []
    print(build(force=args.force or args.verbose, verbose=args.verbose, extra_flags=extra))


if __name__ == "__main__":
    main()
