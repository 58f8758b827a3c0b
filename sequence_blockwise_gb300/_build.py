"""Builds libsp_attn.so in-tree with nvcc for sm_103a (no CMake, no torch
extension machinery): each translation unit is compiled in parallel, then
linked into one shared library next to this file."""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsp_attn.so")

CU_SOURCES = ["sp_api.cu", "attn_tc.cu", "attn_tc_pair.cu", "attn_bwd_tc.cu", "attn_simt.cu", "sp_aux.cu"]
CPP_SOURCES = ["sp_schedule.cpp"]
HEADERS = ["sp_internal.h", "sp_device.cuh", "sp_workspace.h", "sp_tiles.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsp_attn")
    return path


def _inputs():
    files = [os.path.join(CSRC, f) for f in CU_SOURCES + CPP_SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "sp_attn.h"))
    files.append(os.path.abspath(__file__))
    return files


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nv = nvcc()
    common = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]
    procs = []
    objs = []
    for src in CU_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        cmd = [nv, *ARCH, *common, "-lineinfo", "-Xptxas", "-v", "-c", os.path.join(CSRC, src),
               "-o", obj]
        log = open(os.path.join(BUILD, src + ".log"), "w")
        procs.append((src, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
        objs.append(obj)
    for src in CPP_SOURCES:
        obj = os.path.join(BUILD, src + ".o")
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-I", INCLUDE, "-c", os.path.join(CSRC, src),
               "-o", obj]
        log = open(os.path.join(BUILD, src + ".log"), "w")
        procs.append((src, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
        objs.append(obj)
    failed = []
    for src, p, log in procs:
        rc = p.wait()
        log.close()
        if rc != 0:
            failed.append(src)
    if failed:
        msgs = []
        for src in failed:
            with open(os.path.join(BUILD, src + ".log")) as f:
                msgs.append(f"--- {src}\n" + f.read()[-4000:])
        raise RuntimeError("libsp_attn build failed:\n" + "\n".join(msgs))
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call([nv, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    if verbose:
        for src in CU_SOURCES:
            with open(os.path.join(BUILD, src + ".log")) as f:
                print(f.read())
    return LIB


if __name__ == "__main__":
    build(force=True, verbose=True)
    print(LIB)
