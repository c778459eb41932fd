"""Build libmtpspec.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel, then linked into one shared
library with the CUDA runtime linked statically.  ptxas resource usage
(registers, spills, shared memory) is kept in _build/ptxas.log.

variant="bounds" builds the bounds-checked library (-DMTP_BOUNDS: an index
outside its buffer sets MTP_STATUS_BOUNDS and the access is skipped) into
_build_bounds/libmtpspec_bounds.so; the binding loads it when the environment
sets MTP_LIB_VARIANT=bounds.  variant="trace" builds the launch-tracing
library (-DMTP_TRACE: every kernel stamps its start, dependency release and
end on the GPU's global timer; mtp_trace_read) into _build_trace/, loaded
with MTP_LIB_VARIANT=trace.
"""

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(BUILD, "libmtpspec.so")
VARIANTS = {"": (BUILD, LIB, []),
            "bounds": (os.path.join(PKG, "_build_bounds"),
                       os.path.join(PKG, "_build_bounds", "libmtpspec_bounds.so"), ["-DMTP_BOUNDS"]),
            "trace": (os.path.join(PKG, "_build_trace"),
                      os.path.join(PKG, "_build_trace", "libmtpspec_trace.so"), ["-DMTP_TRACE"])}


def library_path(variant=None):
    """The shared library the binding loads: the default build, or the one
    MTP_LIB_VARIANT names."""
    v = os.environ.get("MTP_LIB_VARIANT", "") if variant is None else variant
    if v not in VARIANTS:
        raise RuntimeError("unknown MTP_LIB_VARIANT %r (known: %s)" % (v, ", ".join(repr(k) for k in VARIANTS)))
    return VARIANTS[v][1]
SOURCES = ("api.cu", "draft.cu", "verify.cu", "verify_split.cu", "tc.cu", "attn_tc.cu", "diag.cu", "fused.cu",
           "chain.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmtpspec")
    return exe


def _needs_rebuild(lib):
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "mtpspec.h"), __file__]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force=False, verbose=False, variant=""):
    """Compile and link the library (the default one, or a variant) if any
    source is newer; return its path."""
    build_dir, lib, extra = VARIANTS[variant]
    if not force and not _needs_rebuild(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    flags = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
             "-I", INCLUDE, "-I", CSRC] + ARCH + extra

    def compile_one(src):
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj] + flags
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    log = []
    for src, obj, r in results:
        log.append("==== %s\n%s" % (src, r.stderr))
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s" % (src, r.stderr[-6000:]))
    with open(os.path.join(build_dir, "ptxas.log"), "w") as f:
        f.write("\n".join(log))
    tmp = lib + ".tmp"
    cmd = [nvcc(), "-shared", "-o", tmp] + [o for _, o, _ in results] + ARCH + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s" % r.stderr[-6000:])
    os.replace(tmp, lib)
    if verbose:
        print("built", lib, file=sys.stderr)
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, variant="bounds" if "--bounds" in sys.argv else "")
