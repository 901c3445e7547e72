"""Build the in-tree shared libraries with nvcc.

``_lib/liblora_b300.so`` is the product: every ``csrc/*.cu`` file compiled
for sm_103a only (``-gencode arch=compute_103a,code=sm_103a``) and linked
with the static CUDA runtime, so the library loads on a machine without a
GPU (the C ABI then reports errors instead of launching).
``_lib/liblora_b300_testhooks.so`` is the same sources built with
``-DLORA_TEST_HOOKS``: it adds the test-only entry point of
``include/lora_b300_test_hooks.h``, which lets a test make a device-side
wait run out; nothing but that test loads it.  Run ``python
lora_qlora_linear_fwd_b300/build.py`` (this file imports nothing from the
package, so it also works while the library is missing or stale).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "_lib")
LIBNAME = "liblora_b300.so"
OBJDIR = os.path.join(ROOT, "_build", "obj")
# variant -> (library file, object directory, extra nvcc flags)
VARIANTS = {
    "product": (LIBNAME, OBJDIR, []),
    "testhooks": ("liblora_b300_testhooks.so", os.path.join(ROOT, "_build", "obj_testhooks"),
                  ["-DLORA_TEST_HOOKS"]),
}

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O3",
         "--expt-relaxed-constexpr", "-Xptxas", "-v", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found")
    return exe


def lib_path(variant: str = "product") -> str:
    return os.path.join(LIBDIR, VARIANTS[variant][0])


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                  + glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, obj: str, log_dir: str, extra=()) -> str:
    cmd = [nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    log = os.path.join(log_dir, os.path.basename(src) + ".ptxas.txt")
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr[-6000:]}")
    return obj


def build_variant(variant: str, force: bool = False, jobs: int | None = None) -> str:
    """Compile (if stale) and link one library variant; return its path."""
    libname, objdir, extra = VARIANTS[variant]
    os.makedirs(LIBDIR, exist_ok=True)
    os.makedirs(objdir, exist_ok=True)
    hdrs = _headers()
    work = []
    objs = []
    for src in _sources():
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        objs.append(obj)
        if force or _stale(obj, [src, *hdrs]):
            work.append((src, obj))
    if work:
        jobs = jobs or min(len(work), os.cpu_count() or 4)
        with cf.ThreadPoolExecutor(jobs) as ex:
            futs = [ex.submit(_compile, s, o, objdir, extra) for s, o in work]
            for f in futs:
                f.result()
    out = os.path.join(LIBDIR, libname)
    if force or work or _stale(out, objs):
        cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", out, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    return out


def build(force: bool = False, jobs: int | None = None, verbose: bool = False) -> str:
    """Build every variant; return the product library's path."""
    with cf.ThreadPoolExecutor(len(VARIANTS)) as ex:
        futs = {v: ex.submit(build_variant, v, force, jobs) for v in VARIANTS}
        paths = {v: f.result() for v, f in futs.items()}
    if verbose:
        for p in paths.values():
            print(p)
    return paths["product"]


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
