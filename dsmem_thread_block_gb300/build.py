"""Build libcredit.so in-tree with nvcc for sm_103a.

Each translation unit under csrc/ is compiled in parallel, then linked into
``dsmem_thread_block_gb300/_build/libcredit.so``.  No cmake, one -gencode.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libcredit.so")
# the checked build: the same sources with -DCREDIT_DEBUG (index checks and the
# phase trace), in its own object directory
CHECKED_LIB = os.path.join(BUILD, "libcredit_checked.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    p = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(p):
        return p
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcredit")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    out = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    out += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return out


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps() + [__file__])


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None,
          checked: bool = False) -> str:
    """Compile and link libcredit.so (checked: libcredit_checked.so, with
    -DCREDIT_DEBUG) if any source is newer than it."""
    lib = CHECKED_LIB if checked else LIB
    if not force and not _stale(lib):
        return lib
    objdir = os.path.join(BUILD, "checked") if checked else BUILD
    os.makedirs(objdir, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-Xcompiler", "-Wall", "-I", INCLUDE, "--expt-relaxed-constexpr"]
    if checked:
        flags += ["-DCREDIT_DEBUG"]
    if verbose:
        flags += ["-Xptxas", "-v"]
    flags += list(extra or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        r = subprocess.run([cc, *flags, "-c", src, "-o", obj], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".{os.getpid()}.tmp"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> tuple[str, str]:
    """Both libraries, compiled side by side: (regular, checked)."""
    with cf.ThreadPoolExecutor(max_workers=2) as ex:
        reg = ex.submit(build, force)
        chk = ex.submit(build, force, False, None, True)
        return reg.result(), chk.result()


if __name__ == "__main__":
    if "--checked" in sys.argv:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked=True))
    else:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
