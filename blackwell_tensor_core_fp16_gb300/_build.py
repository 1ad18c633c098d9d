"""Build step for libgemm_f16.so: one nvcc invocation, sm_103a only, in-tree output."""
from __future__ import annotations

import os
import re
import shutil
import subprocess
import tempfile

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
HEADERS = [os.path.join(ROOT, "include", "gemm_f16.h"), os.path.join(ROOT, "include", "gdn.h")]
SOURCES = ["gemm_f16.cu", "gdn.cu"]   # translation units, compiled in parallel
LIB_PATH = os.path.join(PKG_DIR, "libgemm_f16.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
    "-shared",
]


def _nvcc() -> str:
    found = shutil.which("nvcc")
    if found:
        return found
    for cand in ("/usr/local/cuda/bin/nvcc",):
        if os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgemm_f16.so")


def _sources():
    srcs = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))
            if f.endswith((".cu", ".cuh", ".h"))]
    return srcs + HEADERS


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(s) > t for s in _sources())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/gemm_f16.cu and csrc/gdn.cu (in parallel) and link libgemm_f16.so next to
    this file."""
    if not force and not is_stale():
        return LIB_PATH
    tag = f"tmp{os.getpid()}"
    compile_flags = [f for f in NVCC_FLAGS if f != "-shared"]
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(PKG_DIR, f".{os.path.splitext(src)[0]}.{tag}.o")
        cmd = [_nvcc(), *compile_flags, "-c", "-o", obj, os.path.join(CSRC, src)]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append(subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
        objs.append(obj)
    errors, logs = [], []
    for p in procs:
        out, err = p.communicate()
        logs.append(out + err)
        if p.returncode != 0:
            errors.append(f"nvcc failed ({p.returncode}):\n{out}\n{err}")
    try:
        if errors:
            raise RuntimeError("\n".join(errors))
        tmp = LIB_PATH + "." + tag
        res = subprocess.run([_nvcc(), *NVCC_FLAGS, "-o", tmp, *objs], capture_output=True,
                             text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc link failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.unlink(obj)
    if verbose:
        print("".join(logs))
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def ptxas_report() -> dict:
    """Resource usage ptxas reports for every function of the library (nvcc -Xptxas -v): per
    mangled name, its stack frame, spill stores and spill loads in bytes, and, for kernels, the
    registers per thread.  Compiles into a temporary directory; the library is left as it is."""
    compile_flags = [f for f in NVCC_FLAGS if f != "-shared"]
    funcs: dict = {}
    with tempfile.TemporaryDirectory() as tmp:
        procs = []
        for src in SOURCES:
            obj = os.path.join(tmp, os.path.splitext(src)[0] + ".o")
            cmd = [_nvcc(), "-Xptxas=-v", *compile_flags, "-c", "-o", obj,
                   os.path.join(CSRC, src)]
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
        for src, p in procs:
            out, _ = p.communicate()
            if p.returncode != 0:
                raise RuntimeError(f"nvcc failed on {src} ({p.returncode}):\n{out}")
            current = None
            for line in out.splitlines():
                m = re.search(r"Function properties for (\S+)", line)
                if m:
                    current = funcs.setdefault(m.group(1), {"source": src})
                    continue
                m = re.search(r"Compiling entry function '([^']+)'", line)
                if m:
                    current = funcs.setdefault(m.group(1), {"source": src})
                    current["entry"] = True
                    continue
                m = re.search(r"(\d+) bytes stack frame, (\d+) bytes spill stores, "
                              r"(\d+) bytes spill loads", line)
                if m and current is not None:
                    current.update(stack=int(m.group(1)), spill_stores=int(m.group(2)),
                                   spill_loads=int(m.group(3)))
                    continue
                m = re.search(r"Used (\d+) registers", line)
                if m and current is not None:
                    current["registers"] = int(m.group(1))
    return funcs
