"""In-tree build of librlloss.so for sm_103a with nvcc (no cmake, no torch extension).

The translation units are compiled in parallel, then linked into
``ppo_policy_loss_gb300/librlloss.so`` against the shared CUDA runtime (the same
libcudart PyTorch loads, so device pointers and streams are shared).
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "librlloss.so")
SOURCES = ["policy_loss.cu", "advantages.cu", "critic.cu", "status.cu", "lmhead.cu", "lmhead_grad.cu"]
# (object, source, extra flags): policy_loss.cu builds a second time with the
# short-row configuration of the loss kernel.
UNITS = [(src.replace(".cu", ".o"), src, []) for src in SOURCES] + [
    ("policy_loss_short_rows.o", "policy_loss.cu", ["-DRL_SHORT_ROWS"])]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-I" + INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build librlloss.so")
    return p


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "rlloss.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link librlloss.so if any source is newer; return its path."""
    if not force and up_to_date():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(OBJ_DIR, exist_ok=True)
    procs, objs = [], []
    for name, src, extra in UNITS:
        obj = os.path.join(OBJ_DIR, name)
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            print(out.decode(errors="replace"))
        if p.returncode:
            failed.append(" ".join(cmd))
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
            "-Xlinker", "-rpath," + os.path.join(os.path.dirname(os.path.dirname(nvcc)), "lib64")]
    subprocess.check_call(link)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH
