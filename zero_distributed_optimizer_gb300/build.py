"""Build the dopt shared library (libdopt.so) in-tree for sm_103a.

The host file is compiled by g++ and the CUDA file by nvcc, in parallel, then
linked with nvcc.  The output is keyed by a hash of the sources and flags, so
an unchanged tree is not rebuilt.  Usable as a script: ``python -m
zero_distributed_optimizer_gb300.build [--force]``.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libdopt.so")
STAMP = LIB + ".stamp"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
HOST_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-ffp-contract=off", "-fno-fast-math", "-Wall"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-fmad=false",
                     "-Xcompiler", "-fPIC,-O2,-ffp-contract=off,-fno-fast-math"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdopt.so")


def cuda_home() -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc())))


def sources():
    host = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith(".cpp")]
    dev = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith(".cu")]
    hdr = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC)) if f.endswith((".h", ".cuh"))]
    hdr += [os.path.join(INCLUDE, f) for f in sorted(os.listdir(INCLUDE)) if f.endswith(".h")]
    return host, dev, hdr


def source_hash() -> str:
    h = hashlib.sha256()
    host, dev, hdr = sources()
    for path in host + dev + hdr:
        h.update(os.path.basename(path).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    h.update(" ".join(HOST_FLAGS + NVCC_FLAGS).encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def is_current() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(STAMP)):
        return False
    with open(STAMP) as f:
        return f.read().strip() == source_hash()


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libdopt.so if the sources changed; return its path."""
    if not force and is_current():
        return LIB
    host, dev, _ = sources()
    inc = ["-I", INCLUDE, "-I", CSRC, "-I", os.path.join(cuda_home(), "include")]
    with tempfile.TemporaryDirectory(prefix="dopt_build_") as tmp:
        jobs, objs = [], []
        for src in host:
            obj = os.path.join(tmp, os.path.basename(src) + ".o")
            jobs.append(["g++", *HOST_FLAGS, *inc, "-c", src, "-o", obj])
            objs.append(obj)
        for src in dev:
            obj = os.path.join(tmp, os.path.basename(src) + ".o")
            jobs.append([nvcc(), *NVCC_FLAGS, *inc, "-c", src, "-o", obj])
            objs.append(obj)
        procs = [subprocess.Popen(j, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
                 for j in jobs]
        failed = []
        for j, p in zip(jobs, procs):
            out, _ = p.communicate()
            if verbose and out:
                sys.stderr.write(out)
            if p.returncode != 0:
                failed.append((j, out))
        if failed:
            msg = "\n".join(" ".join(j) + "\n" + out for j, out in failed)
            raise RuntimeError(f"libdopt build failed:\n{msg}")
        tmp_lib = os.path.join(tmp, "libdopt.so")
        link = [nvcc(), *ARCH, "-shared", "-o", tmp_lib, *objs]
        res = subprocess.run(link, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("libdopt link failed:\n" + " ".join(link) + "\n" + res.stdout + res.stderr)
        shutil.copyfile(tmp_lib, LIB + ".tmp")
        os.replace(LIB + ".tmp", LIB)
    with open(STAMP, "w") as f:
        f.write(source_hash())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
