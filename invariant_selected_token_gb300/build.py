"""Build the CUDA library librlk.so in place (sm_103a only).

    python -m invariant_selected_token_gb300.build [--force] [--verbose]

Each translation unit is compiled by nvcc in parallel, then linked into
``invariant_selected_token_gb300/librlk.so`` with the CUDA runtime linked
statically.  The contract flags (-ftz=false -prec-div=true -prec-sqrt=true
-fmad=false) keep the compiler from flushing subnormals, approximating
division or fusing multiply-adds on its own: every rounding the numeric
contract names is written explicitly in the source.
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "librlk.so")
INCLUDE = os.path.join(ROOT, "include")

SOURCES = ["rlk_logits.cu", "rlk_logits_mat.cu", "rlk_merge.cu", "rlk_gemm.cu", "rlk_rmsnorm.cu",
           "rlk_api.cu", "rlk_static_ws.cu", "rlk_debug.cu"]
HEADERS = ["rlk_ptx.cuh", "rlk_contract.cuh", "rlk_internal.h"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CONTRACT_FLAGS = ["-ftz=false", "-prec-div=true", "-prec-sqrt=true", "-fmad=false"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-Wall", "--expt-relaxed-constexpr"] + CONTRACT_FLAGS


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def nvcc_version() -> str:
    try:
        out = subprocess.run([nvcc(), "--version"], capture_output=True, text=True, check=True).stdout
        for line in out.splitlines():
            if "release" in line:
                return line.split("release")[-1].strip().replace(",", "").replace(" ", "_")
    except Exception:
        pass
    return "unknown"


def source_digest() -> str:
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    with open(os.path.join(INCLUDE, "rlk.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(NVCC_FLAGS).encode())
    return h.hexdigest()[:16]


def unit_digest(src: str) -> str:
    """Digest of one translation unit's inputs: the source, every shared header, the C
    header and the flags.  Counters taken from a kernel stay valid while it is unchanged."""
    h = hashlib.sha256()
    for name in [src] + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    with open(os.path.join(INCLUDE, "rlk.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(NVCC_FLAGS).encode())
    return "unit-" + h.hexdigest()[:16]


def _compile(src: str, defines, verbose: bool) -> str:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc()] + NVCC_FLAGS + defines + ["-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    digest = source_digest()
    stamp = os.path.join(BUILD, "stamp")
    if not force and os.path.exists(LIB) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return LIB
    os.makedirs(BUILD, exist_ok=True)
    defines = ['-DRLK_GIT_REV="src-%s"' % digest, '-DRLK_NVCC_VERSION="%s"' % nvcc_version()]
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, defines, verbose), SOURCES))
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(digest)
    return LIB


if __name__ == "__main__":
    if "--unit-digest" in sys.argv:
        print(unit_digest(sys.argv[sys.argv.index("--unit-digest") + 1]))
    else:
        print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
