"""Build the C-ABI shared library ``libmoe_b300.so`` in this directory with nvcc for
sm_103a. Each .cu file compiles to an object under ``_build/`` (in parallel), then
they link into one shared library with the CUDA runtime linked statically.

    python -m mixture_experts_layer_102_b300.build [--force] [--ptxas-verbose]
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libmoe_b300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
SOURCES = ["moe_abi.cu", "router.cu", "router_tc.cu", "route_select.cu", "route_fused.cu",
           "reroute.cu",
           "capacity.cu", "combine.cu", "gemm_simt.cu", "gemm_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "moe.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = False) -> str:
    if not force and up_to_date():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I", INCLUDE, "-I", CSRC]
    if ptxas_verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src: str):
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj] + common
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 1)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    failed = False
    for src, _, r in results:
        out = (r.stdout + r.stderr).strip()
        if r.returncode != 0:
            failed = True
            sys.stderr.write(f"--- nvcc failed on {src}\n{out}\n")
        elif out and (ptxas_verbose or not quiet):
            sys.stderr.write(f"--- {src}\n{out}\n")
    if failed:
        raise RuntimeError("CUDA build failed")
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, "-shared"] + ARCH + ["-o", tmp] + [obj for _, obj, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


HOOKS_LIB_PATH = os.path.join(HERE, "libmoe_b300_testhooks.so")


def build_test_hooks(force: bool = False, quiet: bool = False) -> str:
    """The test build of the library (include/moe_test_hooks.h): the product objects
    with gemm_tc.cu recompiled under MOE_TEST_HOOKS, linked as
    ``libmoe_b300_testhooks.so``. Only tests load it."""
    build(force=force, quiet=quiet)
    deps = _deps() + [os.path.join(INCLUDE, "moe_test_hooks.h")]
    if (not force and os.path.exists(HOOKS_LIB_PATH)
            and all(os.path.getmtime(f) <= os.path.getmtime(HOOKS_LIB_PATH) for f in deps)):
        return HOOKS_LIB_PATH
    nvcc = _nvcc()
    obj = os.path.join(BUILD_DIR, "gemm_tc_hooks.o")
    cmd = [nvcc, "-c", os.path.join(CSRC, "gemm_tc.cu"), "-o", obj, "-DMOE_TEST_HOOKS"] + ARCH + \
        ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed on gemm_tc.cu (test hooks):\n" + r.stdout + r.stderr)
    objs = [os.path.join(BUILD_DIR, s.replace(".cu", ".o")) for s in SOURCES if s != "gemm_tc.cu"]
    tmp = HOOKS_LIB_PATH + ".tmp"
    r = subprocess.run([nvcc, "-shared"] + ARCH + ["-o", tmp] + objs + [obj],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, HOOKS_LIB_PATH)
    return HOOKS_LIB_PATH


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, ptxas_verbose=args.ptxas_verbose))
    print(build_test_hooks())


if __name__ == "__main__":
    main()
