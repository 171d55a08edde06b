"""Builds the C-ABI library ``_lib/libmatrixopt.so`` in-tree for sm_103a.

    python -m matrix_optimizers_gb300.build

Each translation unit compiles in parallel with nvcc; the host code is built
with floating-point contraction off so that the owner planner performs exactly
the IEEE operations its definition lists, on x86 and on Arm alike.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB_NAME = "libmatrixopt.so"
SOURCES = ["api.cu", "elementwise.cu", "ns_tc.cu", "ns_fp32.cu", "spectral.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmatrixopt")


def common_flags():
    return ARCH + [
        "-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
        "-Xcompiler", "-fPIC", "-Xcompiler", "-ffp-contract=off", "-Xcompiler", "-O2",
        "-I" + os.path.join(ROOT, "include"),
    ]


def _compile(src, obj, verbose):
    cmd = [nvcc_path(), "-c", os.path.join(CSRC, src), "-o", obj] + common_flags()
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return r.stderr


def lib_path():
    return os.path.join(OUT_DIR, LIB_NAME)


def build(verbose=False, force=False):
    """Compile every CUDA source and link the shared library; returns its path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    target = lib_path()
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))] + \
        [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))]
    if not force and os.path.exists(target):
        t = os.path.getmtime(target)
        if all(os.path.getmtime(d) <= t for d in deps) and os.path.getmtime(__file__) <= t:
            return target
    objs = [os.path.join(OUT_DIR, s.replace(".cu", ".o")) for s in SOURCES]
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        logs = list(ex.map(lambda so: _compile(so[0], so[1], verbose), zip(SOURCES, objs)))
    if verbose:
        for s, log in zip(SOURCES, logs):
            sys.stderr.write(f"--- {s}\n{log}")
    tmp = target + ".tmp"
    cmd = [nvcc_path(), "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "shared"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, target)
    for o in objs:
        os.remove(o)
    return target


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force=True))
