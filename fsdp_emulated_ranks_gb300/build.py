"""Build ``libcr.so`` (the CUDA kernels and the C ABI of include/cr.h) for
sm_103a with nvcc, in-tree under ``fsdp_emulated_ranks_gb300/_build``.

Translation units compile in parallel; the link step produces one shared
library with the CUDA runtime linked statically, so loading it needs no
torch and no CUDA device (the driver is only opened at the first launch).
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libcr.so")
# The checked variant (device-side index checks, csrc/check.cuh), for tests.
CHECKED_DIR = os.path.join(PKG, "_build_checked")
CHECKED_LIB_PATH = os.path.join(CHECKED_DIR, "libcr.so")
CHECKED_FLAGS = ["-DCR_DEVICE_CHECKS", "-rdc=true"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC]
SOURCES = ["api.cu", "api_buckets.cu", "api_optim.cu", "api_range.cu", "launch_util.cu", "k_collectives.cu", "k_fsdp.cu",
           "k_bucket.cu", "k_bucket_fused.cu", "k_fsdp2.cu", "k_accum.cu",
           "k_hsdp.cu", "reducer.cu", "fsdp_noalloc.cu", "check.cu", "plan.cpp",
           "comm.cpp"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcr")


def _inputs() -> list[str]:
    files = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))]
    files.append(os.path.join(INCLUDE, "cr.h"))
    files.append(os.path.abspath(__file__))
    return files


def source_hash() -> str:
    """Hash of every source the library is built from."""
    h = hashlib.sha256()
    for f in _inputs():
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _local_includes(path: str, seen: set) -> None:
    """Files under csrc/ or include/ that `path` includes, transitively."""
    with open(path) as fh:
        for line in fh:
            line = line.strip()
            if not line.startswith("#include \""):
                continue
            name = line.split('"')[1]
            for d in (CSRC, INCLUDE):
                q = os.path.join(d, name)
                if os.path.exists(q) and q not in seen:
                    seen.add(q)
                    _local_includes(q, seen)
                    break


def code_tokens(text: str) -> str:
    """C/C++ source with its comments removed and every run of whitespace
    made one space: what the compiler sees of it, up to the preprocessor.
    String and character literals are kept as they are."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    # keep line structure for preprocessor directives, squeeze the rest
    lines = (" ".join(l.split()) for l in "".join(out).splitlines())
    return "\n".join(l for l in lines if l)


def kernel_hash(tu: str) -> str:
    """Hash of what the kernels of one translation unit are compiled from:
    the code of that file and of the library headers it includes
    (transitively), comments and layout aside, and the compiler flags.  A
    profile of a kernel stays valid while this hash is unchanged; editing a
    comment does not change it."""
    h = hashlib.sha256()
    # the flags without the include paths, which differ between checkouts
    h.update(" ".join(f for f in ARCH + NVCC_FLAGS if not f.startswith("-I")).encode())
    src = os.path.join(CSRC, tu)
    deps: set = set()
    _local_includes(src, deps)
    for f in [src] + sorted(deps, key=os.path.basename):
        h.update(os.path.basename(f).encode())
        with open(f, encoding="utf-8") as fh:
            h.update(code_tokens(fh.read()).encode())
    return h.hexdigest()[:16]


def _dir(checked: bool) -> str:
    return CHECKED_DIR if checked else BUILD_DIR


def _stamp(checked: bool = False) -> str:
    return os.path.join(_dir(checked), "libcr.hash")


def up_to_date(checked: bool = False) -> bool:
    lib = CHECKED_LIB_PATH if checked else LIB_PATH
    if not os.path.exists(lib) or not os.path.exists(_stamp(checked)):
        return False
    with open(_stamp(checked)) as f:
        return f.read().strip() == source_hash()


def _compile(src: str, verbose_ptxas: bool, checked: bool) -> str:
    obj = os.path.join(_dir(checked), os.path.basename(src) + ".o")
    extra = CHECKED_FLAGS if checked else []
    cmd = [nvcc()] + ARCH + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
    if src.endswith(".cpp"):
        cmd = [nvcc()] + ["-x", "c++"] + NVCC_FLAGS + ["-c", src, "-o", obj]
    elif verbose_ptxas:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    if verbose_ptxas and res.stderr:
        sys.stderr.write(res.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, checked: bool = False) -> str:
    """Compile libcr.so if it is missing or stale; return its path.
    checked=True builds the variant with device-side index checks into its
    own directory (tests only)."""
    lib = CHECKED_LIB_PATH if checked else LIB_PATH
    if not force and up_to_date(checked):
        return lib
    os.makedirs(_dir(checked), exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, checked), srcs))
    tmp = lib + ".tmp.%d" % os.getpid()
    extra = ["-rdc=true"] if checked else []
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static"] + extra + ["-o", tmp] + objs
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    with open(_stamp(checked), "w") as f:
        f.write(source_hash())
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
