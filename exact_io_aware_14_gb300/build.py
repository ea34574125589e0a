"""Builds the CUDA library in-tree: exact_io_aware_14_gb300/_build/libattn_sm103.so
(and, on request, build variants under _build/<variant>/).

Each .cu file is compiled by its own nvcc process (in parallel) for sm_103a
only, then linked into one shared object with the CUDA runtime linked
statically.  The driver API entry point the library needs
(cuTensorMapEncodeTiled) is looked up at run time, so no libcuda is needed
at link time and the library loads on a machine without a GPU.
"""
import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libattn_sm103.so")
NVCC = os.environ.get("NVCC", "nvcc")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                               + glob.glob(os.path.join(ROOT, "include", "*.h"))) + [__file__]


# Build variants: the same sources with preprocessor switches, each in its own
# directory.  "exp2poly<K>": the prefill softmax computes every K-th pair of
# exponentials with the software exp2 (csrc/exp2_poly.cuh) instead of MUFU.
VARIANTS = {"exp2poly%d" % k: ["-DATTN_EXP2_POLY=%d" % k] for k in (2, 4, 8, 16)}


def variant_lib_path(name: str) -> str:
    return os.path.join(OUT_DIR, name, "libattn_sm103.so")


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build_variant(name: str, force: bool = False, verbose: bool = False) -> str:
    """Builds the library with the switches of VARIANTS[name] into
    _build/<name>/libattn_sm103.so (same exported interface)."""
    defines = VARIANTS[name]
    lib = variant_lib_path(name)
    if not force and up_to_date(lib):
        return lib
    return _build(os.path.dirname(lib), lib, defines, verbose, False)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    return _build(OUT_DIR, LIB, [], verbose, ptxas_info)


def _build(out_dir, lib, defines, verbose, ptxas_info):
    os.makedirs(out_dir, exist_ok=True)
    srcs = _sources()
    objs = [os.path.join(out_dir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    extra = (["-Xptxas", "-v"] if ptxas_info else []) + list(defines)

    def compile_one(so):
        s, o = so
        cmd = [NVCC] + FLAGS + extra + ["-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return s, r

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, zip(srcs, objs)))
    for s, r in results:
        if verbose or ptxas_info or r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s" % os.path.basename(s))
    tmp = lib + ".tmp%d" % os.getpid()
    cmd = [NVCC] + ARCH + ["-shared", "-Xcompiler", "-fPIC", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc link failed")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    names = [a for a in sys.argv[1:] if not a.startswith("--")]
    if names:
        for n in names:
            print(build_variant(n, force="--force" in sys.argv, verbose=True))
    else:
        print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv))
