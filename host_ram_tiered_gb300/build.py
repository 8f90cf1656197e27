"""Build libkvo.so (the CUDA library behind include/kvo.h) in-tree with nvcc.

Every translation unit is compiled for sm_103a only, in parallel, then
linked into ``host_ram_tiered_gb300/libkvo.so``.  No cmake, no torch
extension machinery: the library has a plain C ABI.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libkvo.so")

# The decode kernels are instantiated in one unit per K/V dtype, head_dim and
# mode (decode_k_*.cu), the slowest units first, so that they compile in parallel.
DECODE_KERNEL_UNITS = [f"decode_k_{m}{dt}_{d}.cu" for m, dts in (("sp_", ("f16", "bf16")), ("", ("f16", "bf16", "q8_0")))
                       for dt in dts for d in (128, 64)]
SOURCES = DECODE_KERNEL_UNITS + ["prefill_tc.cu", "prefill_mma.cu", "kvo_abi.cu", "swap_gather.cu", "decode.cu",
                                 "decode_f16.cu", "decode_bf16.cu", "decode_q8_0.cu", "decode_noalloc.cu",
                                 "append.cu", "sparse_rows.cu", "vmm.cu", "selftest.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("kvo_internal.cuh", "decode_impl.cuh", "decode_dispatch.cuh", "sync.cuh")] + \
    [os.path.join(ROOT, "include", "kvo.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvo")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    procs, objs = [], []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [path] + HEADERS):
            cmd = [cc] + ARCH + NVCC_FLAGS + ["-c", path, "-o", obj]
            if ptxas_info:
                cmd.insert(1, "-Xptxas=-v")
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif (verbose or ptxas_info) and text.strip():
            print(text, file=sys.stderr)
    if failed:
        msg = "\n".join(f"--- {s}\n{t}" for s, t in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    if force or _stale(LIB_PATH, objs):
        tmp = LIB_PATH + ".tmp%d" % os.getpid()
        cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB_PATH)
