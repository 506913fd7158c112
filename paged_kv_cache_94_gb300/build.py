"""Build libpa.so in-tree with nvcc for sm_103a.

The translation units compile in parallel into paged_kv_cache_94_gb300/_build/
and link into paged_kv_cache_94_gb300/lib/libpa.so. Only one -gencode is used:
  -gencode arch=compute_103a,code=sm_103a
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libpa.so")
INCLUDE = os.path.join(ROOT, "include")

SOURCES = [
    "pa_api.cu",
    "pa_cache_write.cu",
    "pa_decode_bf16_d128.cu",
    "pa_decode_bf16_d64.cu",
    "pa_decode_int8_d128.cu",
    "pa_decode_int8_d64.cu",
    "pa_decode_int4_d128.cu",
    "pa_decode_int4_d64.cu",
    "pa_decode_bf16_mq.cu",
    "pa_decode_int8_mq_d128.cu",
    "pa_decode_int8_mq_d64.cu",
    "pa_decode_int4_mq_d128.cu",
    "pa_decode_int4_mq_d64.cu",
    "pa_share.cu",
    "pa_selftest.cu",
    "pa_decode_noalloc.cu",
    "pa_block_copy.cu",
    "pa_probe.cu",
    "pa_alloc.cpp",
]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    cand = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cand, "bin", "nvcc")
    return path if os.path.exists(path) else (shutil.which("nvcc") or "nvcc")


def _stamp() -> str:
    """Machine + hash of every source the library is built from."""
    h = hashlib.sha256(platform.machine().encode())
    files = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC))
    files += sorted(os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE))
    files.append(os.path.abspath(__file__))
    for f in files:
        h.update(open(f, "rb").read())
    return h.hexdigest()


def _compile(src: str, verbose_ptxas: bool, build_dir: str, defines: list) -> str:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *[f"-D{d}" for d in defines], "-c",
           os.path.join(CSRC, src), "-o", obj]
    if verbose_ptxas:
        cmd[1:1] = ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int = 0,
          out_dir: str = "", defines: tuple = ()) -> str:
    """Compile (if stale) and return the path of libpa.so.

    out_dir/defines build a variant elsewhere (tuning: e.g. defines
    ("PA_BF16_D128_NW=8",) change the warps per CTA); the default is the
    in-tree library the package loads.
    """
    lib_dir = out_dir or LIBDIR
    build_dir = os.path.join(out_dir, "_build") if out_dir else BUILD
    lib = os.path.join(lib_dir, "libpa.so")
    stamp_path = os.path.join(lib_dir, "BUILD_STAMP")
    stamp = _stamp() + ":" + ",".join(defines)
    if not force and os.path.exists(lib) and os.path.exists(stamp_path) and \
            open(stamp_path).read() == stamp:
        return lib
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(lib_dir, exist_ok=True)
    jobs = jobs or min(len(SOURCES), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose_ptxas, build_dir, list(defines)),
                           SOURCES))
    tmp = lib + f".{os.getpid()}.tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp_path, "w") as f:
        f.write(stamp)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))
