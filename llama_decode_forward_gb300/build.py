"""Builds libllmdecode.so in-tree with nvcc for sm_103a (GB300)."""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libllmdecode.so")
# Variant with the phase trace compiled in (-DLLM_TRACE): same ABI, the step
# kernel also records per-CTA phase timestamps readable with llm_trace_read.
TRACE_DIR = os.path.join(OUT_DIR, "trace")
TRACE_LIB = os.path.join(TRACE_DIR, "libllmdecode_trace.so")
# Variant with device-side index checks (-DLLM_CHECKED): same ABI; a failed
# check skips the access and the call returns LLM_ERR_CHECK.
CHECKED_DIR = os.path.join(OUT_DIR, "checked")
CHECKED_LIB = os.path.join(CHECKED_DIR, "libllmdecode_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              f"-I{os.path.join(ROOT, 'include')}"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.isabs(c) and os.path.exists(c) or not os.path.isabs(c)):
            return c
    return "nvcc"


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(ROOT, "include", "llm.h")]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(s) <= t for s in _inputs())


def compile_command(src: str, obj: str, trace: bool = False, verbose: bool = False,
                    checked: bool = False) -> list[str]:
    """The nvcc command that compiles one source for sm_103a."""
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, *(["-DLLM_TRACE"] if trace else []), *(["-DLLM_CHECKED"] if checked else []),
           "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def link_command(objs: list[str], out: str) -> list[str]:
    """The nvcc command that links the objects into the shared library."""
    return [_nvcc(), *ARCH, "-shared", "-o", out, *objs]


def build(force: bool = False, verbose: bool = False, trace: bool = False, checked: bool = False) -> str:
    """Compile every .cu under csrc/ (in parallel) and link the shared library
    (with trace=True, the phase-trace variant; with checked=True, the
    index-checked variant)."""
    if trace and checked:
        raise ValueError("one variant at a time")
    lib, out_dir = (TRACE_LIB, TRACE_DIR) if trace else (CHECKED_LIB, CHECKED_DIR) if checked else (LIB, OUT_DIR)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.splitext(os.path.basename(src))[0] + ".o")
        cmd = compile_command(src, obj, trace, verbose, checked)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, len(sources()))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    r = subprocess.run(link_command(objs, tmp), capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, trace="--trace" in sys.argv,
                checked="--checked" in sys.argv))
