"""Build libsyn.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit compiles in parallel; the result is
``decoder_token_step_gb300/_build/libsyn.so``. A unit is recompiled only when it or a header
changed. Set ``SYN_PTXAS_VERBOSE=1`` to print register and shared-memory use per kernel.
"""
from __future__ import annotations

import hashlib
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libsyn.so")

SOURCES = ["archdef.cpp", "sha256.cpp", "runtime.cpp", "k_gemv.cu", "k_gemm_tc.cu", "k_attn.cu", "k_attn_tc.cu",
           "k_misc.cu", "attn_static.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.isabs(c) and os.path.exists(c) or not os.path.isabs(c)):
            return c
    return "nvcc"


def _flags() -> list:
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
                "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    if os.environ.get("SYN_PTXAS_VERBOSE"):
        f += ["-Xptxas", "-v"]
    return f


def _headers_digest() -> str:
    h = hashlib.sha256()
    for d in (CSRC, os.path.join(ROOT, "include")):
        for name in sorted(os.listdir(d)):
            if name.endswith((".h", ".cuh")):
                with open(os.path.join(d, name), "rb") as f:
                    h.update(name.encode() + f.read())
    return h.hexdigest()


def _unit_key(src: str, flags: list, hdr: str) -> str:
    with open(os.path.join(CSRC, src), "rb") as f:
        body = f.read()
    return hashlib.sha256(body + " ".join(flags).encode() + hdr.encode()).hexdigest()[:24]


def build(verbose: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    flags = _flags()
    hdr = _headers_digest()
    nvcc = _nvcc()

    def compile_one(src: str) -> str:
        key = _unit_key(src, flags, hdr)
        obj = os.path.join(OUT, f"{os.path.splitext(src)[0]}.{key}.o")
        if os.path.exists(obj):
            return obj
        tmp = obj + f".{os.getpid()}.tmp"
        cmd = [nvcc] + flags + ["-c", os.path.join(CSRC, src), "-o", tmp]
        if src.endswith(".cpp"):
            cmd = [nvcc] + flags + ["-x", "cu", "-c", os.path.join(CSRC, src), "-o", tmp]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or os.environ.get("SYN_PTXAS_VERBOSE"):
            sys.stderr.write(r.stderr)
        os.replace(tmp, obj)
        return obj

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    link_key = hashlib.sha256("".join(objs).encode()).hexdigest()[:24]
    stamp = os.path.join(OUT, "libsyn.link")
    if os.path.exists(LIB) and os.path.exists(stamp) and open(stamp).read() == link_key:
        return LIB
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(link_key)
    # drop stale objects of earlier builds
    keep = set(os.path.basename(o) for o in objs)
    for name in os.listdir(OUT):
        if name.endswith(".o") and name not in keep:
            try:
                os.remove(os.path.join(OUT, name))
            except OSError:
                pass
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
