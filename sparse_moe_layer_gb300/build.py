"""Build libmoe_gb300.so in-tree for sm_103a (nvcc, one -gencode, parallel TUs)."""
from __future__ import annotations

import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoe_gb300.so")
SOURCES = ["moe_api.cu", "moe_route.cu", "moe_gemm.cu", "moe_gemm_decode.cu", "moe_gemm_mx.cu"]
HEADERS = ["moe_device.cuh", "moe_internal.h"]
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xptxas", "-v"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(ROOT, "include", "moe_gb300.h")]
    return any(os.path.getmtime(d) > t for d in deps)


GEMM_LAUNCH_REGS = 168  # must match GemmCfg<...>::LAUNCH_REGS (setmaxnreg budget)


def _check_gemm_registers(log_path: str) -> None:
    """The prefill GEMMs move registers between warpgroups with setmaxnreg; the
    split balances only if each kernel launches with exactly 168 registers."""
    import re
    text = open(log_path).read()
    found = re.findall(r"Compiling entry function '(_ZN3moe15moe_gemm_kernelILb[01]E[^']*)'.*?Used (\d+) registers", text,
                       re.S)
    if len(found) != 2 or any(int(n) != GEMM_LAUNCH_REGS for _, n in found):
        raise RuntimeError(f"prefill GEMMs compiled to {[n for _, n in found]} registers, expected {GEMM_LAUNCH_REGS}")
    if "setmaxnreg" in text and "ignored" in text:
        raise RuntimeError("ptxas ignored setmaxnreg in a prefill GEMM")


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [nvcc, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        with open(os.path.join(BUILD, src + ".log"), "w") as f:
            f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr[-4000:]}")
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    _check_gemm_registers(os.path.join(BUILD, "moe_gemm.cu.log"))
    tmp = LIB + ".tmp"
    r = subprocess.run([nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-o", tmp, *objs],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, LIB)
    if verbose:
        for src in SOURCES:
            print(open(os.path.join(BUILD, src + ".log")).read())
    return LIB


if __name__ == "__main__":
    build(force=True, verbose=True)
