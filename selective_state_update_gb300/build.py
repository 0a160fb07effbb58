"""Build libssu.so (the CUDA kernels and the C ABI) in-tree with nvcc.

    python -m selective_state_update_gb300.build [-v]

Translation units are compiled in parallel for sm_103a only; the result goes to
``selective_state_update_gb300/_build/libssu.so``.  A content hash of the
sources and flags decides whether anything needs rebuilding.
"""
from __future__ import annotations

import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libssu.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-Wall", "-I", INCLUDE, "-I", CSRC]
SOURCES = ["ssu_api.cpp", "ssu_onetoken.cu", "ssu_packed.cu", "ssu_packed_long.cu", "ssu_replay_f32.cu", "ssu_replay_f16.cu",
           "ssu_replay_bf16.cu", "ssu_copy.cu", "ssu_shadow.cu", "ssu_ssd.cu", "ssu_ssd_tc.cu", "ssu_verify.cu"]
HEADERS = ["ssu_internal.h", "ssu_device.cuh", "ssu_replay.cuh", "ssu_ssd_params.h", "ssu_verify.h"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; libssu needs the CUDA toolkit to build")
    return cand


def _digest(extra_flags) -> str:
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    with open(os.path.join(INCLUDE, "ssu.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(ARCH + COMMON + list(extra_flags)).encode())
    return h.hexdigest()


def build(verbose: bool = False, force: bool = False, extra_flags=(), out_dir: str = OUT_DIR) -> str:
    """Compile every translation unit and link ``libssu.so`` into ``out_dir``;
    returns its path."""
    os.makedirs(out_dir, exist_ok=True)
    lib_path = os.path.join(out_dir, "libssu.so")
    stamp = os.path.join(out_dir, "libssu.sha256")
    digest = _digest(extra_flags)
    if not force and os.path.exists(lib_path) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == digest:
                return lib_path
    nvcc = _nvcc()
    flags = ARCH + COMMON + list(extra_flags) + (["-Xptxas", "-v"] if verbose else [])

    def compile_one(name):
        src = os.path.join(CSRC, name)
        obj = os.path.join(out_dir, name + ".o")
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {name}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"linking libssu.so failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    with open(stamp, "w") as f:
        f.write(digest)
    return lib_path


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
