"""Build libmoe_ptpc.so in-tree from csrc/*.cu with nvcc for sm_103a.

Each translation unit compiles in parallel, then one link step produces the
shared library (static CUDA runtime, only the moe_* C symbols exported).
A stamp file records the host architecture and a hash of the sources and
flags, so a library built on another machine is never reused.

Variant "check" builds libmoe_ptpc_check.so with -DMOE_CHECK: every
data-dependent index (expert ids, row maps) is validated where it is used, and
a bad one sets an error bit instead of going out of bounds. The binding loads
it when MOE_LIBRARY_VARIANT=check.
"""

import hashlib
import os
import platform
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libmoe_ptpc.so"

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH_FLAGS + [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
    "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE,
]


VARIANTS = {"": ([], LIB_NAME, "_build"),
            "check": (["-DMOE_CHECK"], "libmoe_ptpc_check.so", "_build_check")}


def library_path(variant=""):
    return os.path.join(PKG, VARIANTS[variant][1])


def _nvcc():
    exe = shutil.which("nvcc")
    if exe is None:
        cand = "/usr/local/cuda/bin/nvcc"
        if os.path.exists(cand):
            exe = cand
    if exe is None:
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to "
                           "build the MoE kernels")
    return exe


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith(".cu"))


def _stamp(extra_flags):
    h = hashlib.sha256()
    h.update(platform.machine().encode())
    h.update(" ".join(NVCC_FLAGS + list(extra_flags)).encode())
    for d in (CSRC, INCLUDE):
        for f in sorted(os.listdir(d)):
            p = os.path.join(d, f)
            if os.path.isfile(p):
                h.update(f.encode())
                with open(p, "rb") as fh:
                    h.update(fh.read())
    return h.hexdigest()


def build(force=False, extra_flags=(), verbose=False, jobs=None, variant=""):
    """Compile and link the library (or its variant); returns its path."""
    vflags, _, vdir = VARIANTS[variant]
    extra_flags = list(vflags) + list(extra_flags)
    build_dir = os.path.join(PKG, vdir)
    lib = library_path(variant)
    stamp_file = os.path.join(build_dir, "stamp")
    stamp = _stamp(extra_flags)
    if (not force and os.path.exists(lib) and os.path.exists(stamp_file)
            and open(stamp_file).read() == stamp):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    srcs = _sources()
    objs = [os.path.join(build_dir, os.path.basename(s)[:-3] + ".o")
            for s in srcs]

    def compile_one(pair):
        src, obj = pair
        cmd = [nvcc] + NVCC_FLAGS + list(extra_flags) + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n"
                               f"{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)

    with ThreadPoolExecutor(max_workers=jobs or min(len(srcs),
                                                    os.cpu_count() or 4)) as ex:
        list(ex.map(compile_one, zip(srcs, objs)))
    tmp = lib + ".tmp"
    cmd = [nvcc] + ARCH_FLAGS + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp_file, "w") as fh:
        fh.write(stamp)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))
