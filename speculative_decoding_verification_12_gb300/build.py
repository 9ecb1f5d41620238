"""Builds the CUDA library in-tree for sm_103a (GB300) with nvcc.

The shared object lands next to this file as libspecverify.so.  It links the CUDA runtime
dynamically, so a process that already loaded PyTorch's libcudart.so.13 shares it.
"""
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libspecverify.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def deps():
    out = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    out.append(os.path.join(os.path.dirname(HERE), "include", "spec_verify.h"))
    return out


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libspecverify.so unless it is newer than every source.  Each translation unit
    (one per logits dtype and scheme, plus the entry points) compiles in its own nvcc process,
    in parallel; one link makes the library."""
    if not force and os.path.exists(LIB):
        t = os.path.getmtime(LIB)
        if all(os.path.getmtime(p) <= t for p in deps()):
            return LIB
    tag = f"{os.getpid()}"
    objs, procs = [], []
    for src in sources():
        obj = os.path.join(CSRC, os.path.basename(src)[:-3] + f".{tag}.o")
        cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-c", "-o", obj, src]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        objs.append(obj)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = False
    for src, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0 or verbose:
            sys.stderr.write(out)
        failed = failed or pr.returncode != 0
    try:
        if failed:
            raise RuntimeError("nvcc failed building libspecverify.so")
        tmp = LIB + f".tmp{tag}"
        res = subprocess.run([nvcc(), *ARCH, "-shared", "-cudart", "shared", "-Xlinker",
                              "-rpath,/usr/local/cuda/lib64", "-o", tmp, *objs], capture_output=True, text=True)
        if res.returncode != 0:
            sys.stderr.write(res.stdout + res.stderr)
            raise RuntimeError("linking libspecverify.so failed")
        os.replace(tmp, LIB)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
