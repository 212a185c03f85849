"""Build ``libpa.so`` (the C-ABI CUDA library) in-tree, for sm_103a only.

Each translation unit is compiled by nvcc in parallel, then linked into one
shared library with the CUDA runtime linked statically.  No CMake, no torch
extension machinery: the library has a plain C ABI (see include/pa.h).
"""
import os
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBRARY = os.path.join(HERE, "libpa.so")
# decode.cu comes first among the slow units so that it starts first.
SOURCES = ["decode_mma_shared.cu", "decode_mma_plain.cu", "decode_fma.cu", "decode_simt.cu", "decode.cu", "pa_api.cu",
           "cache_ops.cu", "block_manager.cpp", "simulator.cpp", "shared_plan.cpp"]
HEADERS = ["pa_common.cuh", "pa_internal.h", "decode_kernels.h", "decode_merge.cuh", "decode_plan.cuh", "decode_simt.cuh",
           "decode_mma.cuh", "decode_tc.cuh", "decode_fma.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _stale():
    if not os.path.exists(LIBRARY):
        return True
    t = os.path.getmtime(LIBRARY)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS] + [os.path.join(INCLUDE, "pa.h"), __file__]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libpa.so if missing or older than its sources; return its path."""
    if not (force or _stale()):
        return LIBRARY
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-lineinfo", "-I", INCLUDE, "-Xcompiler", "-fPIC,-O2,-Wall",
              "--expt-relaxed-constexpr"] + ARCH
    with tempfile.TemporaryDirectory(prefix="pa_build_") as tmp:
        procs, objs = [], []
        for src in SOURCES:
            obj = os.path.join(tmp, src + ".o")
            cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj] + common
            if src.endswith(".cpp"):
                cmd += ["-x", "cu"]
            if verbose:
                cmd += ["-Xptxas", "-v"]
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
            objs.append(obj)
        failed = []
        for src, p in procs:
            out, _ = p.communicate()
            if p.returncode != 0 or verbose:
                sys.stderr.write(out.decode(errors="replace"))
            if p.returncode != 0:
                failed.append(src)
        if failed:
            raise RuntimeError("nvcc failed for: " + ", ".join(failed))
        tmp_lib = LIBRARY + ".tmp.%d" % os.getpid()
        link = [nvcc, "-shared", "-o", tmp_lib] + objs + ARCH + ["-cudart", "static", "-lpthread", "-ldl", "-lrt"]
        subprocess.run(link, check=True)
        os.replace(tmp_lib, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
