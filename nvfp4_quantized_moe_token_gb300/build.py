"""Build libnvfp4moe.so (the C-ABI CUDA library) in-tree for sm_103a.

Each .cu file compiles in parallel to an object, then one nvcc link makes
the shared library.  Only sm_103a code is generated.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libnvfp4moe.so")
SOURCES = ["api.cu", "quantize.cu", "dequantize.cu", "route.cu", "gemm.cu", "gemm_bf16.cu", "combine.cu",
           "noalloc.cu"]
HEADERS = ["common.cuh", "fastdiv.cuh", "nvfp4_encode.cuh", "route_topk.cuh", "kernels.h", os.path.join("..", "..", "include", "nvfp4moe.h")]

NVCC = os.environ.get("NVCC", shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc")
FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-std=c++17", "-lineinfo",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr",
]


def _newest_input():
    paths = [os.path.join(CSRC, s) for s in SOURCES] + [os.path.join(CSRC, h) for h in HEADERS]
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


def _compile(src, verbose):
    obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [NVCC, *FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force=False, verbose=False):
    """Compile the library if any source changed; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    objs = [o for o, _ in results]
    if verbose:
        for (_, log), src in zip(results, SOURCES):
            if log.strip():
                print(f"--- {src}\n{log}")
    tmp = LIB + f".tmp{os.getpid()}"
    # exported symbols: the extern "C" entry points (visibility default there)
    cmd = [NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp, *objs,
           "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
