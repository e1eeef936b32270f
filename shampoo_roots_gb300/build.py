"""Build libprecond.so in-tree with nvcc for sm_103a (no cmake, one translation unit)."""
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libprecond.so")
SOURCES = ["precond.cu"]
FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
         "-Xcompiler", "-fPIC", "-shared"]


def nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources_newer_than(target):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    root = os.path.dirname(HERE)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(root, "include", "precond.h")]
    return any(os.path.getmtime(p) > t for p in deps if os.path.exists(p))


def build(force=False, verbose=False):
    if not force and not sources_newer_than(OUT):
        return OUT
    tmp = OUT + ".tmp"
    cmd = [nvcc()] + FLAGS + ["-o", tmp] + [os.path.join(CSRC, s) for s in SOURCES]
    if verbose:
        print(" ".join(cmd))
    subprocess.run(cmd, check=True, cwd=CSRC)
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force=True, verbose=True))
