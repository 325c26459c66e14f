"""Build the CUDA library (liblsv.so) in-tree for sm_103a with nvcc.

Each translation unit compiles in parallel; the shared library links against
the shared CUDA runtime, the same one PyTorch loads.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(OUT_DIR, "liblsv.so")
SOURCES = ["api.cu", "route.cu", "permute.cu", "ffn.cu", "combine.cu", "accept.cu", "prefetch.cu", "lmhead.cu", "attention.cu", "policy.cu", "draft.cu", "skinny.cu", "cache.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _cuda_home(nvcc: str) -> str:
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False, extra_flags: list[str] | None = None,
          out_dir: str | None = None) -> str:
    """Compile into out_dir (default: the package's _lib/) and return the library path."""
    nvcc = _nvcc()
    odir = out_dir or OUT_DIR
    lib_path = os.path.join(odir, "liblsv.so")
    os.makedirs(odir, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    headers.append(os.path.join(INCLUDE, "lsv.h"))
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC,
                    "--expt-relaxed-constexpr"] + list(extra_flags or [])
    if verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        s = os.path.join(CSRC, src)
        o = os.path.join(odir, src.replace(".cu", ".o"))
        if force or _stale(o, [s] + headers):
            cmd = [nvcc, "-c", s, "-o", o + ".tmp.o"] + flags
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
            os.replace(o + ".tmp.o", o)
            if verbose:
                sys.stderr.write(r.stderr)
        return o

    with cf.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or _stale(lib_path, objs):
        lib64 = os.path.join(_cuda_home(nvcc), "lib64")
        tmp = lib_path + ".%d.tmp" % os.getpid()
        cmd = [nvcc, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "shared", "-Xlinker",
                                                            "-rpath," + lib64]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
