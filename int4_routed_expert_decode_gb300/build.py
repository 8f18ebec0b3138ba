"""Build the CUDA library ``libmoe_gb300.so`` in-tree with nvcc (sm_103a only).

Each ``csrc/*.cu`` compiles to an object under ``_build/`` in parallel (only
when it or a header is newer than its object), then nvcc links the shared
library next to this file.  The CUDA runtime is linked statically.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmoe_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(ROOT, "include", "*.h"))


def _compile(src: str, ptxas_verbose: bool, obj_dir: str = OBJ,
             defines: tuple = ()) -> tuple[str, str]:
    obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
    newest = max([os.path.getmtime(src)] + [os.path.getmtime(h) for h in _headers()])
    if os.path.exists(obj) and os.path.getmtime(obj) >= newest and not ptxas_verbose:
        return obj, ""
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *[f"-D{d}" for d in defines], "-c", src, "-o", obj]
    if ptxas_verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose: bool = False, ptxas_verbose: bool = False, jobs: int | None = None,
          defines: tuple = (), lib_path: str = LIB, obj_dir: str = OBJ) -> str:
    """Build the library; `defines` (macro names) select an instrumented
    variant, which then needs its own `obj_dir` and `lib_path`."""
    os.makedirs(obj_dir, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    jobs = jobs or min(len(sources), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(jobs) as ex:
        results = list(ex.map(lambda s: _compile(s, ptxas_verbose, obj_dir, defines), sources))
    objs = [o for o, _ in results]
    if ptxas_verbose or verbose:
        for o, log in results:
            if log:
                sys.stderr.write(log)
    if os.path.exists(lib_path) and \
            os.path.getmtime(lib_path) >= max(os.path.getmtime(o) for o in objs):
        return lib_path
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(lib_path))
    os.close(fd)
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        os.unlink(tmp)
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(verbose=True, ptxas_verbose="-v" in sys.argv))
