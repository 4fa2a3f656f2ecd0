"""Build libnvfp4.so (the C-ABI library of include/nvfp4.h) for sm_103a.

Each CUDA translation unit is compiled in parallel with nvcc, then linked into
fp4_gemm_nvfp4_gb300/_build/libnvfp4.so (in-tree, git-ignored).  With
debug=True the same sources are built with NVFP4_BOUNDS_CHECK into
fp4_gemm_nvfp4_gb300/_build_debug/libnvfp4_debug.so: every output store
checks its bytes against the range the call declared for that buffer and is
skipped and counted when outside (include/nvfp4_testing.h).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libnvfp4.so")
OUT_DIR_DEBUG = os.path.join(HERE, "_build_debug")
LIB_DEBUG = os.path.join(OUT_DIR_DEBUG, "libnvfp4_debug.so")
SOURCES = ["api.cu", "quantize.cu", "gemm.cu", "dequantize.cu", "quantize_noalloc.cu"]
HEADERS = ["device_common.cuh", "kernels.h", "bounds.cuh"]
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
         "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall", "-Xcompiler", "-fvisibility=hidden", "-I", os.path.join(ROOT, "include")]


def _newest_input():
    paths = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    paths += [os.path.join(ROOT, "include", h) for h in ("nvfp4.h", "nvfp4_testing.h")]
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile and link the library (or, with debug, its bounds-checked build)
    if it is missing or out of date."""
    out_dir, lib = (OUT_DIR_DEBUG, LIB_DEBUG) if debug else (OUT_DIR, LIB)
    if debug:
        extra_flags = (*extra_flags, "-DNVFP4_BOUNDS_CHECK")
    os.makedirs(out_dir, exist_ok=True)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input():
        return lib
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [NVCC, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed on {failed}")
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.run([NVCC, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *objs, "-o", tmp],
                   check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else [], debug="--debug" in sys.argv))
