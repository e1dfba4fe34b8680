"""Build libpagedkv.so in-tree for sm_103a with nvcc (translation units compiled in parallel)."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG, "libpagedkv.so")
SOURCES = ["pkv_api.cu", "pkv_attn.cu", "pkv_attn_cols.cu", "pkv_attn_tc.cu", "pkv_cache_ops.cu"]
HEADERS = ["pkv_device.cuh", "pkv_internal.h", "pkv_attn_common.cuh", "pkv_cols.cuh", "pkv_tcgen05.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libpagedkv needs the CUDA toolkit to build")


def _stale(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "pkv.h"),
                                                                  os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build_library(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
                  out: str | None = None, defines=(), build_dir: str | None = None) -> str:
    """Compile every .cu to an object in _build/, link libpagedkv.so next to this file.

    ``out``/``defines``/``build_dir`` build a variant elsewhere (e.g. the test build with
    -DPKV_TEST_HOOKS, or other pipeline depths via -DPKV_STAGES=...; a variant is rebuilt when any
    source is newer than it, so give each set of defines its own ``out`` and ``build_dir``); the
    default build is the in-tree library the package loads.
    """
    variant = out is not None
    out = out or LIB_PATH
    bdir = build_dir or BUILD_DIR
    if not force and not _stale(out):
        return out
    nvcc = nvcc_path()
    os.makedirs(bdir, exist_ok=True)
    common = [nvcc, "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC,-fvisibility=hidden",
              "-I", INCLUDE, "-I", CSRC, *[f"-D{d}" for d in defines]]
    if ptxas_info:
        common += ["-Xptxas", "-v"]
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = common + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    logs = []
    failed = []
    for src, p in procs:
        text, _ = p.communicate()
        logs.append(text.decode(errors="replace"))
        if p.returncode != 0:
            failed.append(src)
    log_text = "".join(logs)
    with open(os.path.join(bdir, "compile.log"), "w") as f:
        f.write(log_text)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}:\n{log_text}")
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, out)
    if verbose:
        print(log_text, file=sys.stderr)
    return out


if __name__ == "__main__":
    build_library(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
