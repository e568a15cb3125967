"""Build ``libpagedkv.so`` (the C-ABI CUDA library) in-tree for sm_103a.

Each ``csrc/*.cu`` is compiled in parallel with nvcc for
``-gencode arch=compute_103a,code=sm_103a`` and linked with a static CUDA
runtime into ``paged_kv_cache_172_gb300/libpagedkv.so``.  Objects go to
``paged_kv_cache_172_gb300/_build/``.  Rebuilds only what changed.
"""
import glob
import hashlib
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libpagedkv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall", "-I", INCLUDE, "-I", CSRC]


def nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedkv")
    return path


def _headers_mtime():
    hs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    return max(os.path.getmtime(h) for h in hs)


def _compile(src, extra, obj_dir):
    obj = os.path.join(obj_dir, os.path.basename(src) + ".o")
    if (os.path.exists(obj) and os.path.getmtime(obj) >= os.path.getmtime(src)
            and os.path.getmtime(obj) >= _headers_mtime()):
        return obj, None
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        return obj, f"$ {' '.join(cmd)}\n{r.stdout}\n{r.stderr}"
    return obj, r.stderr if "warning" in r.stderr.lower() else None


def build(verbose: bool = False, extra_flags=(), out=None, sources=None) -> str:
    """Compile and link.  ``extra_flags`` (e.g. -D tuning macros) build a
    variant with its own object directory; ``out`` names its library path;
    ``sources`` (file names in csrc/) limits a variant to those files."""
    extra_flags = tuple(extra_flags)
    lib = out or LIB
    obj_dir = OBJ_DIR
    if extra_flags:
        tag = hashlib.sha256(" ".join(extra_flags).encode()).hexdigest()[:10]
        obj_dir = os.path.join(OBJ_DIR, "variant_" + tag)
    os.makedirs(obj_dir, exist_ok=True)
    if sources is None:
        srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    else:
        srcs = [os.path.join(CSRC, s) for s in sources]
    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(lambda s: _compile(s, list(extra_flags), obj_dir), srcs))
    errors = [msg for _, msg in results if msg and "error" in msg.lower()]
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    if verbose:
        for _, msg in results:
            if msg:
                print(msg, file=sys.stderr)
    objs = [o for o, _ in results]
    if (os.path.exists(lib)
            and all(os.path.getmtime(lib) >= os.path.getmtime(o) for o in objs)):
        return lib
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n$ {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True, extra_flags=tuple(sys.argv[1:])))
