"""Builds libdsa.so in-tree for sm_103a with nvcc (no cmake, no torch).

    python -m sparse_attention_decode_paged_gb300.build

Every CUDA source is compiled in parallel with one -gencode
(arch=compute_103a,code=sm_103a) and linked into
sparse_attention_decode_paged_gb300/libdsa.so.  A stamp next to the library
records the machine and a hash of sources and flags; a stale or foreign
library (for example one built on another CPU architecture) is rebuilt.
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
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
LIB = os.path.join(PKG, "libdsa.so")
STAMP = LIB + ".stamp"
# read-only stream probe (not part of the DSA path; only the benchmark loads it)
PROBE_SRC = os.path.join(PKG, "probe", "read_stream.cu")
PROBE_LIB = os.path.join(PKG, "libdsa_probe.so")

GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-Xptxas", "-warn-spills"] + GENCODE


def cuda_home() -> str:
    for cand in (os.environ.get("CUDA_HOME"), os.environ.get("CUDA_PATH"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return cand
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(nvcc))
    raise RuntimeError("nvcc not found (set CUDA_HOME)")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cu", ".cpp")))


def _digest() -> str:
    h = hashlib.sha256()
    h.update(platform.machine().encode())
    h.update(" ".join(NVCC_FLAGS).encode())
    for d in (CSRC, INCLUDE, os.path.dirname(PROBE_SRC)):
        for f in sorted(os.listdir(d)):
            with open(os.path.join(d, f), "rb") as fh:
                h.update(f.encode())
                h.update(fh.read())
    return h.hexdigest()


def up_to_date() -> bool:
    if not (os.path.exists(LIB) and os.path.exists(STAMP) and os.path.exists(PROBE_LIB)):
        return False
    with open(STAMP) as f:
        return f.read().strip() == _digest()


def build(verbose: bool = False, force: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    nvcc = os.path.join(cuda_home(), "bin", "nvcc")
    obj_dir = os.path.join(PKG, "_build", platform.machine())
    os.makedirs(obj_dir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, "-c", src, "-o", obj, "-I", INCLUDE, "-I", CSRC] + NVCC_FLAGS
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    def build_probe():
        tmp = PROBE_LIB + ".tmp"
        cmd = [nvcc, "-shared", PROBE_SRC, "-o", tmp] + NVCC_FLAGS
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on the read probe:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, PROBE_LIB)

    srcs = sources()
    with cf.ThreadPoolExecutor(max(1, min(len(srcs) + 1, os.cpu_count() or 1))) as ex:
        probe = ex.submit(build_probe)
        objs = list(ex.map(compile_one, srcs))
        probe.result()
    tmp = LIB + ".tmp"
    cmd = [nvcc, "-shared", "-o", tmp] + objs + GENCODE
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(STAMP, "w") as f:
        f.write(_digest())
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
