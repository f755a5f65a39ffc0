"""Build the in-tree CUDA library liblagb300.so for sm_103a with nvcc.

Each .cu under csrc/ compiles in parallel to an object (one -gencode,
compute_103a -> sm_103a, -lineinfo), then nvcc links them into a shared
library with the static CUDA runtime.  No torch, no cmake: the same command
works on x86_64 (cross-compile, no GPU) and on the aarch64 GPU hosts.
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIB = os.path.join(HERE, "liblagb300.so")
OBJDIR = os.path.join(HERE, "_build")
# the bounds-checking build (LA_CHECK_BOUNDS): index checks in the tensor-core
# kernels record failures in the device error word instead of accessing
CHECKED_LIB = os.path.join(HERE, "liblagb300_checked.so")
CHECKED_OBJDIR = os.path.join(HERE, "_build_checked")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I", CSRC, "-I", INCLUDE]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "la.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, extra=(), checked: bool = False) -> str:
    """Build liblagb300.so, or with checked=True liblagb300_checked.so (the
    same sources with LA_CHECK_BOUNDS defined); returns the library's path."""
    lib, objdir = (CHECKED_LIB, CHECKED_OBJDIR) if checked else (LIB, OBJDIR)
    if checked:
        extra = (*extra, "-DLA_CHECK_BOUNDS")
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps():
        return lib
    nvcc = _nvcc()
    os.makedirs(objdir, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = lib + ".tmp.%d" % os.getpid()
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-cudart", "static", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    extra = [a for a in sys.argv[1:] if a.startswith("-X") or a.startswith("--")]
    extra = [a for a in extra if a not in ("--force", "--checked")]
    print(build(force="--force" in sys.argv, verbose=True, extra=extra,
                checked="--checked" in sys.argv))
