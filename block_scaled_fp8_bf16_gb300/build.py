"""Builds libfp8blk.so in-tree with nvcc for sm_103a.

Each .cu file compiles to an object in parallel, then one link produces the
shared library next to this file.  ptxas resource usage of every kernel is
kept in _build/ptxas.log; the build fails if any kernel spills to local
memory or uses a stack frame (the register-budget check).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import re
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libfp8blk.so")
SOURCES = ["api.cu", "quant.cu", "gemm_w8a8.cu", "gemm_w8a8_pair.cu", "gemm_w8a8_mx.cu", "gemm_w8a16.cu",
           "gemm_w8a16_decode.cu", "gemv.cu"]
HEADERS = ["ptx.cuh", "decode.cuh", "quant.cuh", "internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
         "-I", INCLUDE, "-I", CSRC, "-Xptxas", "-v", "-Werror", "all-warnings"]


def nvcc_path() -> str:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found")
    return p


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "fp8blk.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile(nvcc, src):
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc, *ARCH, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, r.returncode, r.stdout + r.stderr, cmd


# Kernels that rebalance registers between warpgroups with setmaxnreg: the
# split is computed for exactly this many registers per thread at launch, so
# any other count must stop the build (a split larger than the launch
# allocation would wait forever).
SETMAXNREG_KERNELS = {"w8a8_pair_kernel": 168}


def check_resources(log: str) -> list[str]:
    """Kernels whose ptxas report shows spill stores/loads or a stack frame,
    or a register count other than the one their register split assumes."""
    bad = []
    current = None
    for line in log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
        m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m and current and any(int(v) for v in m.groups()):
            bad.append(f"{current}: {line.strip()}")
        m = re.search(r"Used (\d+) registers", line)
        if m and current:
            for name, regs in SETMAXNREG_KERNELS.items():
                if name in current and int(m.group(1)) != regs:
                    bad.append(f"{current}: {m.group(1)} registers, register split assumes {regs}")
    return bad


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(nvcc, s), SOURCES))
    log = []
    for src, obj, rc, out, cmd in results:
        log.append(f"== {src}\n{out}")
        if rc != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{out}")
    log_text = "\n".join(log)
    with open(os.path.join(BUILD_DIR, "ptxas.log"), "w") as f:
        f.write(log_text)
    bad = check_resources(log_text)
    if bad:
        raise RuntimeError("kernels spill or use a stack frame:\n" + "\n".join(bad))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *[r[1] for r in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}{r.stderr}")
    os.replace(tmp, LIB_PATH)
    if verbose:
        print(log_text, file=sys.stderr)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
