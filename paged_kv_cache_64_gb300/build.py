"""Build the CUDA library libpa.so (sm_103a) in-tree.

Every translation unit under csrc/ is compiled in parallel (nvcc for the .cu
files: decode, tensor-core decode, E4M3 decode, cascade, cache write and block
copy; g++ for the .cpp files: the block allocator and the prefix-caching
pool) and linked by nvcc into paged_kv_cache_64_gb300/_build/libpa.so.  The CUDA runtime is linked
statically, so the library only needs the driver at run time.
"""
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libpa.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cu", ".cpp", ".cuh", ".h")))


def _compile_cmd(src, obj):
    if src.endswith(".cu"):
        return [_nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
                "-Xcompiler", "-Wall", "-I", INCLUDE, "-c", src, "-o", obj]
    return ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-Wextra", "-I", INCLUDE,
            "-I", os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include"),
            "-c", src, "-o", obj]


def is_stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = sources() + [os.path.join(INCLUDE, "pa.h"), __file__]
    return any(os.path.getmtime(s) > t for s in deps)


def build(force=False, verbose=False):
    """Compile and link; returns the path of libpa.so."""
    if not force and not is_stale():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    units = [s for s in sources() if s.endswith((".cu", ".cpp"))]
    procs = []
    for src in units:
        obj = os.path.join(OUT_DIR, os.path.basename(src) + ".o")
        cmd = _compile_cmd(src, obj)
        if verbose:
            print(" ".join(cmd))
        procs.append((src, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                 stderr=subprocess.STDOUT)))
    objs, errors = [], []
    for src, obj, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            errors.append(f"{os.path.basename(src)}:\n{out.decode(errors='replace')}")
        elif verbose and out:
            print(out.decode(errors="replace"))
        objs.append(obj)
    if errors:
        raise RuntimeError("libpa build failed:\n" + "\n".join(errors))
    tmp = LIB + ".tmp"
    link = [_nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    p = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if p.returncode != 0:
        raise RuntimeError("libpa link failed:\n" + p.stdout.decode(errors="replace"))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
