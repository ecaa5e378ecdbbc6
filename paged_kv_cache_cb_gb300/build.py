"""Build libcbattn.so in-tree for sm_103a (GB300).

Each translation unit compiles in its own process, in parallel; the objects are
then linked into one shared library next to this file.  No cmake, no torch
extension machinery: plain nvcc and g++.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libcbattn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def _compile(src, extra):
    obj = os.path.join(BUILD, src + ".o")
    path = os.path.join(CSRC, src)
    if src.endswith(".cu"):
        cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
               "-Xcompiler", "-fPIC", "-c", path, "-o", obj, *extra]
    else:
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-c", path, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, obj, r.returncode, r.stdout + r.stderr, cmd


def build(verbose=False, ptxas_info=False):
    """Compile every source under csrc/ and link libcbattn.so.  Returns the path."""
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    srcs = sources()
    with ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda s: _compile(s, extra), srcs))
    failed = [r for r in results if r[2] != 0]
    for src, _, rc, out, cmd in results:
        if verbose or rc != 0 or ptxas_info:
            sys.stderr.write(f"--- {src} (rc={rc})\n{out}")
    if failed:
        raise RuntimeError("build failed: " + ", ".join(r[0] for r in failed))
    objs = [r[1] for r in results]
    tmp = LIB + ".tmp"
    link = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lstdc++"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv))
