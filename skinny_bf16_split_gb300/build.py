"""Build the decode-projection library (libdep_projection.so) for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library next to this file (``_build/``).  Only one architecture is
generated: ``-gencode arch=compute_103a,code=sm_103a``.  No fast-math: FP32
FMA/addition order and denormals are kept exactly as written.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libdep_projection.so")
SOURCES = ["api.cpp", "tma.cpp", "splitk_fma.cu", "tc_gemm.cu", "tc_split.cu", "tc_wide.cu", "tc_cluster.cu", "tc_xm.cu", "mma_rows.cu", "rows_gemv.cu", "staging.cu", "probe.cu"]
HEADERS = ["internal.h", "ptx.cuh", "exchange.cuh", "cluster.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def _flags(extra=()):
    return [*ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
            "-I", INCLUDE, "-I", CSRC, *extra]


DEBUG_DIR = os.path.join(HERE, "_build_debug")


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile every translation unit and link the library; return its path.

    debug=True builds the bounds-checked variant (-DDEP_DEBUG) into _build_debug/:
    every kernel checks each index into y, the plan's workspace and shared
    memory before using it, records DEP_DEV_BOUNDS in the status word and skips
    the access if it is out of range."""
    out_dir = DEBUG_DIR if debug else OUT_DIR
    lib_path = os.path.join(out_dir, "libdep_projection.so")
    if debug:
        extra_flags = ("-DDEP_DEBUG", *extra_flags)
    os.makedirs(out_dir, exist_ok=True)
    deps = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    deps.append(os.path.join(INCLUDE, "dep_projection.h"))
    newest = max(os.path.getmtime(p) for p in deps)
    if not force and os.path.exists(lib_path) and os.path.getmtime(lib_path) >= newest and (debug or not extra_flags):
        return lib_path
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(out_dir, src + ".o")
        cmd = [nvcc, *_flags(extra_flags), "-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cpp"):
            cmd[1:1] = ["-x", "cu"]  # host-only code, still built by nvcc for one toolchain
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else (), debug="--debug" in sys.argv))
