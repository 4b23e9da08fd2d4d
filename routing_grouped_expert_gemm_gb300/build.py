"""Build the CUDA libraries in-tree (sm_103a):

  _lib/libmoe_gb300.so          the product: the C ABI of include/moe.h
  _lib/libmoe_gb300_testing.so  test hooks only (include/moe_testing.h): one-tile
                                probes that pin tensor-core encodings on the GPU

Each translation unit is compiled in parallel with nvcc
(-gencode arch=compute_103a,code=sm_103a -lineinfo -O3) and linked into a
shared library with the CUDA runtime linked statically, so the libraries load
without a GPU (the CPU tests check their exports) and need no libcuda at link
time (the TMA encoder is fetched through the runtime's driver entry point).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB_DIR = os.path.join(HERE, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libmoe_gb300.so")
TESTING_LIB_PATH = os.path.join(LIB_DIR, "libmoe_gb300_testing.so")
TRACE_LIB_PATH = os.path.join(LIB_DIR, "libmoe_gb300_trace.so")
DEBUG_LIB_PATH = os.path.join(LIB_DIR, "libmoe_gb300_dbg.so")
SOURCES = ["api.cu", "router.cu", "schedule.cu", "megakernel.cu", "mxfp8.cu", "route_static.cu", "backward.cu"]
TESTING_SOURCES = ["probe_mx.cu", "probe_pair.cu", "probe_mn.cu", "probe_tma3d.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, verbose: bool, ptxas_v: bool, defines=(), obj_dir: str = OBJ) -> str:
    obj = os.path.join(obj_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
           *[f"-D{d}" for d in defines], "-c", os.path.join(CSRC, src), "-o", obj]
    if ptxas_v:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
    if verbose or ptxas_v:
        sys.stderr.write(r.stderr)
    return obj


def _stale(lib_path: str) -> bool:
    if not os.path.exists(lib_path):
        return True
    t = os.path.getmtime(lib_path)
    inc = os.path.join(HERE, "..", "include")
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(inc, f) for f in os.listdir(inc)]
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def _link(objs, lib_path):
    tmp = lib_path + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", *objs, "-o", tmp, "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stderr)
    os.replace(tmp, lib_path)


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False, trace: bool = False,
          debug_log: bool = False) -> str:
    """Build the library (and, for the plain build, the test-hook library
    beside it); trace=True builds the MOE_TRACE variant (per-CTA wait timers
    in the persistent kernel) as _lib/libmoe_gb300_trace.so instead;
    debug_log=True the MOE_DEBUG_LOG variant (per-CTA progress records and
    bounds checks written to host memory) as _lib/libmoe_gb300_dbg.so."""
    lib_path = TRACE_LIB_PATH if trace else (DEBUG_LIB_PATH if debug_log else LIB_PATH)
    obj_dir = OBJ + ("_trace" if trace else ("_dbg" if debug_log else ""))
    with_testing = not trace and not debug_log
    if not force and not _stale(lib_path) and not (with_testing and _stale(TESTING_LIB_PATH)):
        return lib_path
    os.makedirs(obj_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    defines = ("MOE_TRACE",) if trace else (("MOE_DEBUG_LOG",) if debug_log else ())
    srcs = SOURCES + (TESTING_SOURCES if with_testing else [])
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = dict(zip(srcs, ex.map(lambda s: _compile(s, verbose, ptxas_v, defines, obj_dir), srcs)))
    _link([objs[s] for s in SOURCES], lib_path)
    if with_testing:
        _link([objs[s] for s in TESTING_SOURCES], TESTING_LIB_PATH)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_v="-v" in sys.argv, trace="--trace" in sys.argv,
                debug_log="--debug-log" in sys.argv))
