"""Build the CUDA library libmoe_gb300.so in-tree for sm_103a.

Each translation unit is compiled by nvcc in parallel, then linked into a
shared library with the CUDA runtime linked statically (the library loads
without a GPU or a driver; the driver is reached at run time).
"""
import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(HERE, "csrc")
INC = os.path.join(ROOT, "include")
OBJ = os.path.join(HERE, "_build")
LIB_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIB_DIR, "libmoe_gb300.so")

SOURCES = ["api.cu", "gate.cu", "permute.cu", "gemm.cu", "gemm_block.cu", "act_quant.cu",
           "unpermute.cu", "ep.cu", "gemm_nvfp4.cu", "pipeline.cu", "gemm_wide.cu",
           "gemm_nvfp4_wide.cu"]
# every header beside the sources is a rebuild input (a new one cannot be missed)
HEADERS = sorted(f for f in os.listdir(SRC) if f.endswith((".cuh", ".h")))

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr",
    "-I" + INC, "-I" + SRC,
]


def nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_gb300.so")


def _newest_input():
    files = [os.path.join(SRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(INC, "moe_gb300.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


# "compiled" or "reused": what the last build() call did (so a log can tell a
# fresh compile of the sources from a library left by an earlier build)
last_action = None


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    global last_action
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        last_action = "reused"
        return LIB
    os.makedirs(OBJ, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(OBJ, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *NVCC_FLAGS, *extra, "-c", os.path.join(SRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for (_, log) in results:
            if log.strip():
                print(log)
    objs = [o for o, _ in results]
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *objs, "-o", tmp,
           "-cudart", "static", "-Xcompiler", "-fvisibility=hidden"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    last_action = "compiled"
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose=True, ptxas_info="-v" in sys.argv))
