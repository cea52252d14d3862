"""Build the dopt shared library (libdopt.so) in-tree for sm_103a.

The host file is compiled by g++ and the CUDA file by nvcc, in parallel, then
linked with nvcc.  The output is keyed by a hash of the sources and flags, so
an unchanged tree is not rebuilt.  Usable as a script: ``python -m
zero_distributed_optimizer_gb300.build [--force] [--checked]``.
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
# The test build with the kernels' device-side index checks compiled in
# (DOPT_DEVICE_CHECKS, see dopt_device_checks in dopt.h).
CHECKED_LIB = os.path.join(PKG, "libdopt_checked.so")
CHECKED_FLAGS = ["-DDOPT_DEVICE_CHECKS=1"]

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


def source_hash(extra=()) -> str:
    h = hashlib.sha256()
    host, dev, hdr = sources()
    for path in host + dev + hdr:
        h.update(os.path.basename(path).encode())
        with open(path, "rb") as f:
            h.update(f.read())
    h.update(" ".join(HOST_FLAGS + NVCC_FLAGS + list(extra)).encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def is_current(lib: str = LIB, extra=()) -> bool:
    stamp = lib + ".stamp"
    if not (os.path.exists(lib) and os.path.exists(stamp)):
        return False
    with open(stamp) as f:
        return f.read().strip() == source_hash(extra)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile libdopt.so (or, with checked, the test build
    libdopt_checked.so) if the sources changed; return its path."""
    lib, extra = (CHECKED_LIB, CHECKED_FLAGS) if checked else (LIB, [])
    if not force and is_current(lib, extra):
        return lib
    host, dev, _ = sources()
    inc = ["-I", INCLUDE, "-I", CSRC, "-I", os.path.join(cuda_home(), "include")]
    with tempfile.TemporaryDirectory(prefix="dopt_build_") as tmp:
        jobs, objs = [], []
        for src in host:
            obj = os.path.join(tmp, os.path.basename(src) + ".o")
            jobs.append(["g++", *HOST_FLAGS, *extra, *inc, "-c", src, "-o", obj])
            objs.append(obj)
        for src in dev:
            obj = os.path.join(tmp, os.path.basename(src) + ".o")
            jobs.append([nvcc(), *NVCC_FLAGS, *extra, *inc, "-c", src, "-o", obj])
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
        shutil.copyfile(tmp_lib, lib + ".tmp")
        os.replace(lib + ".tmp", lib)
    with open(lib + ".stamp", "w") as f:
        f.write(source_hash(extra))
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, checked="--checked" in sys.argv))
