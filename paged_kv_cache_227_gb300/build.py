"""Builds the library in-tree: ``paged_kv_cache_227_gb300/libpagedattn.so``.

Each CUDA translation unit is compiled for sm_103a only, in parallel, then
linked with the host allocator into one shared library (static CUDA runtime,
no torch symbols).  Objects go to ``_build/`` beside this file.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(HERE, "libpagedattn.so")
OBJDIR = os.path.join(HERE, "_build")

CU_SOURCES = ["pool.cu", "append.cu", "decode.cu"]
CPP_SOURCES = ["alloc.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        path = os.path.join(cand, "bin", "nvcc") if cand else ""
        if path and os.path.exists(path):
            return path
    return "nvcc"


def _sources():
    srcs = [os.path.join(CSRC, f) for f in CU_SOURCES + CPP_SOURCES]
    deps = srcs + [os.path.join(CSRC, "pa_internal.h"), os.path.join(INCLUDE, "pa.h")]
    return srcs, deps


def up_to_date():
    if not os.path.exists(OUT):
        return False
    _, deps = _sources()
    t = os.path.getmtime(OUT)
    return all(os.path.getmtime(d) <= t for d in deps)


def build(force=False, verbose=False, extra_nvcc=()):
    """Compile and link; returns the path of the shared library."""
    if not force and up_to_date():
        return OUT
    os.makedirs(OBJDIR, exist_ok=True)
    nvcc = _nvcc()
    procs, objs = [], []
    for f in CU_SOURCES:
        obj = os.path.join(OBJDIR, f + ".o")
        cmd = [nvcc, *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
               "-I", INCLUDE, "-I", CSRC, *extra_nvcc, "-c", os.path.join(CSRC, f), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    for f in CPP_SOURCES:
        obj = os.path.join(OBJDIR, f + ".o")
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-I", INCLUDE, "-c", os.path.join(CSRC, f), "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((cmd, text))
        elif verbose and text:
            sys.stdout.write(text)
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + t for c, t in failed)
        raise RuntimeError("library build failed:\n" + msg)
    tmp = OUT + ".tmp"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + " ".join(link) + "\n" + r.stdout + r.stderr)
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
